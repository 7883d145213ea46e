"""The C-ABI library loads and exports every function include/*.h declares;
host-side argument checks return their status codes without touching a
device (no compute calls here)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from serving_sparse_mla_gb300 import binding, build
    build.build()
    return binding.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(sparse_mla_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "sparse_mla_fwd" in names and "sparse_mla_decode" in names and "sparse_mla_fwd_varlen" in names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_header():
    from serving_sparse_mla_gb300 import binding
    assert set(declared_functions()) <= set(binding.SIGNATURES)


def test_status_strings(lib):
    for code in range(7):
        s = lib.sparse_mla_status_string(code).decode()
        assert s.startswith("SPARSE_MLA_")
    assert lib.sparse_mla_status_string(99).decode() == "SPARSE_MLA_UNKNOWN_STATUS"


def _fwd(lib, **kw):
    a = dict(q=16, kv=16, idx=16, scale=0.1, out=16, lse=16, s_q=4, s_kv=8, h_q=8, d_qk=576, d_v=512,
             topk=128, stream=None)
    a.update(kw)
    return lib.sparse_mla_fwd(a["q"], a["kv"], a["idx"], a["scale"], a["out"], a["lse"], a["s_q"], a["s_kv"],
                              a["h_q"], a["d_qk"], a["d_v"], a["topk"], a["stream"])


def test_host_validation_codes(lib):
    assert _fwd(lib, d_qk=512) == 2
    assert _fwd(lib, d_v=576) == 2
    assert _fwd(lib, h_q=0) == 1
    assert _fwd(lib, topk=0) == 1
    assert _fwd(lib, s_q=-1) == 1
    assert _fwd(lib, q=None) == 1
    assert _fwd(lib, out=None) == 1
    assert _fwd(lib, lse=None) == 1
    assert _fwd(lib, q=24) == 1      # not 16-byte aligned
    assert _fwd(lib, idx=18) == 1    # not 4-byte aligned


def test_causal_validation(lib):
    def causal(**kw):
        a = dict(q=16, kv=16, scale=0.1, out=16, lse=16, s_q=4, s_kv=8, h_q=8, d_qk=576, d_v=512, stream=None)
        a.update(kw)
        return lib.sparse_mla_fwd_causal(a["q"], a["kv"], a["scale"], a["out"], a["lse"], a["s_q"], a["s_kv"],
                                         a["h_q"], a["d_qk"], a["d_v"], a["stream"])
    assert causal(d_qk=512) == 2
    assert causal(d_v=256) == 2
    assert causal(h_q=0) == 1
    assert causal(s_q=-1) == 1
    assert causal(s_kv=-1) == 1
    assert causal(q=None) == 1
    assert causal(out=None) == 1
    assert causal(q=24) == 1      # not 16-byte aligned


def test_varlen_and_decode_validation(lib):
    st = lib.sparse_mla_fwd_varlen(16, 16, 16, None, None, 1, 0.1, 16, 16, 4, 4, 8, 576, 512, 64, None)
    assert st == 1
    st = lib.sparse_mla_fwd_varlen(16, 16, 16, 16, 16, 1, 0.1, 16, 16, 4, 4, 8, 576, 256, 64, None)
    assert st == 2
    st = lib.sparse_mla_decode(16, 16, 16, 16, 16, 0.1, 16, 16, 2, 3, 8, 576, 512, 64, 0, 4, 4, None, 0, None)
    assert st == 1   # page_size 0
    st = lib.sparse_mla_decode(16, 16, None, 16, 16, 0.1, 16, 16, 2, 3, 8, 576, 512, 64, 64, 4, 4, None, 0, None)
    assert st == 1   # missing block table
    st = lib.sparse_mla_decode(16, 16, 16, 16, 16, 0.1, 16, 16, 2, 3, 8, 576, 512, 64, 64, 4, 1 << 30, None, 0,
                               None)
    assert st == 1   # num_blocks * page_size overflows int32


def test_workspace_size_rejects_bad_shapes(lib):
    assert lib.sparse_mla_decode_workspace_size(0, 6, 8, 512, 2048) == 0
    assert lib.sparse_mla_decode_workspace_size(4, 6, 8, 256, 2048) == 0
