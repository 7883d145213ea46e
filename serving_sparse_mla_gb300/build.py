"""Build step: compiles the CUDA sources into the in-tree shared library
``libsparse_mla_gb300.so`` for sm_103a with nvcc (no cmake, one translation
unit, one -gencode)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libsparse_mla_gb300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
SOURCES = ["sparse_mla_api.cu"]
DEPS = ["sparse_mla_api.cu", "fwd_kernel.cuh", "bwd_kernel.cuh", "indexer_kernel.cuh", "ptx.cuh"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def nvcc_command(out_path: str = LIB_PATH, extra=()) -> list:
    return [nvcc_path(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
            "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE,
            *extra, "-o", out_path] + [os.path.join(CSRC, s) for s in SOURCES]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, d) for d in DEPS] + [os.path.join(INCLUDE, "sparse_mla.h")]
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if any source is newer than it; returns its path."""
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp)
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
