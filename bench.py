"""Benchmark of the DSA sparse-MLA forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 1..5]

A step is one sparse_mla_fwd call (one pass of the whole hot path) over the
mid-prefill workload of "feat: add XTuner TileLang sparse MLA backend"
(Performance, Isolated sparse MLA forward): s_q = s_kv = 2119, 8 TP-local
query heads, d_qk = 576, d_v = 512, topk = 2048, BF16 Q/KV, causal index
lists padded with -1.  Inputs are seeded synthetic (mla_inputs.config(2)).

Timing: W untimed warm-up steps, then K timed steps bracketed by a barrier
and a device synchronise.  Before every timed step a 256 MB buffer is
written so the step starts with a cold L2 (the inputs are smaller than L2);
each step's kernel is timed with CUDA events on the launching stream and the
sum over the K steps is the device time (max over ranks).  `value` is the
nominal-FLOP throughput 2*s_q*h_q*topk*(576+512) summed over ranks; the
line also carries us/call, gathered-KV GB/s and % of the per-shape roofline.
With N > 1 (torchrun, one process per GPU) every rank runs its own replica
of the workload: weak scaling, no collective on the data path.

--impl reference times the float64 CPU oracle (test infrastructure) on the
host cores instead, on the same workload, as the baseline arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KV_ROW_BYTES = 576 * 2


# ----------------------------------------------------------------------------- helpers

def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bwd", action="store_true",
                    help="time the backward (dq, dkv) on a prefill config (1-4); nominal FLOPs "
                         "2*(3*576 + 2*512) per (token, head, top-k entry), bytes per valid entry = "
                         "1152 gathered + 2304 of fp32 dkv reduction")
    ap.add_argument("--causal", action="store_true",
                    help="time the indices-free causal entry point on the q/kv of a dense prefill config (1-3); "
                         "FLOPs and bytes then count every causal position")
    ap.add_argument("--fp8", action="store_true",
                    help="time the paged decode (config 5) over its cache written as FP8 slots (512 e4m3 codes, four "
                         "fp32 tile scales, 64 bf16 rope values: 656 B per row) through sparse_mla_decode_fp8")
    ap.add_argument("--indexer", action="store_true",
                    help="time the DSA indexer + top-k (dsa_indexer_topk; config 5: dsa_indexer_topk_paged) that "
                         "produces the index lists, on the token shape of config 1-5 with 64 indexer heads of "
                         "width 128; FLOPs "
                         "2*64*128 per scored (row, visible position)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="profiling aid for the dense prefill configs (1-3): s_q = s_kv = TOKENS with the "
                         "config's heads, list pattern and seed (a smaller case of the same kernel)")
    ap.add_argument("--no-all-configs", action="store_true",
                    help="skip the per-workload records of all five forward workloads that the default forward "
                         "run adds under the key 'configs'")
    ap.add_argument("--clock-log", default=None,
                    help="directory for the nvidia-smi clock CSV of the run (default: the system temp dir)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "fwd": ("fwd_kernel.cuh", "ptx.cuh", "sparse_mla_api.cu"),
    "bwd": ("bwd_kernel.cuh", "fwd_kernel.cuh", "ptx.cuh", "sparse_mla_api.cu"),
    "idx": ("indexer_kernel.cuh", "fwd_kernel.cuh", "ptx.cuh", "sparse_mla_api.cu"),
}


def kernel_source_hash(kind: str = "fwd") -> str:
    """Hash of the sources a kernel family is built from (fwd, bwd, idx)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "serving_sparse_mla_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config: int, kind: str = "fwd"):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources (else None)."""
    name = {"fwd": f"fwd_kernel_config{config}_ncu.txt", "bwd": f"bwd_kernel_config{config}_ncu.txt",
            "idx": f"dsa_indexer_config{config}_ncu.txt"}[kind]
    path = os.path.join(ROOT, "profiles", name)
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha") != kernel_source_hash(kind):
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class NvmlClockSampler:
    """SM clock, power and clock-event reasons of this process's GPU, read
    through NVML (read-only queries) every ~2 ms by a thread that samples only
    while the timed region runs.  The NVML device is found by PCI bus id, so
    CUDA_VISIBLE_DEVICES remapping does not matter."""
    NVML_CLOCK_SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        import ctypes
        import threading
        import torch
        self.ok = False
        self.samples = []
        self._run = threading.Event()
        self._stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            pr = torch.cuda.get_device_properties(device)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                uuid = f"GPU-{pr.uuid}".encode()
                if lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(uuid), ctypes.byref(h)) != 0:
                    return
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) != 0:
                return
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            return
        self.lib, self.h, self.max_mhz, self.reasons_fn = lib, h, mx.value, reasons_fn
        self.ctypes = ctypes
        self.ok = True
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def _read(self):
        c = self.ctypes
        clk, mw, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, c.byref(clk)) != 0:
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(mw))
        self.reasons_fn(self.h, c.byref(rs))
        return clk.value, mw.value / 1000.0, rs.value

    def _loop(self):
        while not self._stop.is_set():
            if not self._run.wait(timeout=0.05):
                continue
            r = self._read()
            if r is not None and self._run.is_set():
                self.samples.append(r)
            time.sleep(0.002)

    def start(self):
        if self.ok:
            self._run.set()

    def stop(self):
        if not self.ok:
            return None
        self._run.clear()
        self._stop.set()
        self.thread.join(timeout=2)
        if not self.samples:
            return None
        reasons = set()
        for _, _, bits in self.samples:
            for b, name in self.REASONS.items():
                if bits & b:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[0] for x in self.samples), "sm_max_mhz": self.max_mhz,
                "power_w_median": round(statistics.median(x[1] for x in self.samples), 1),
                "samples": len(self.samples), "source": "nvml, 2 ms", "reasons": sorted(reasons)}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons every 200 ms into a CSV beside the
    run (a record of the whole run; the NVML sampler covers the timed region)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_dir: str):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.log_dir = log_dir

    def start(self):
        try:
            os.makedirs(self.log_dir, exist_ok=True)
            self.path = os.path.join(self.log_dir, f"clocks_rank{self.gpu}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "source": "nvidia-smi, 200 ms", "reasons": sorted(reasons)}


def max_over_ranks(vals, dist, device=None):
    """Elementwise max of per-rank timings (identity with one rank)."""
    if dist is None:
        return [float(v) for v in vals]
    import torch
    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_tflops(flops_per_step: float, steps: int, world: int, max_total_ms: float) -> float:
    """Units processed by all ranks (each runs its own replica) / slowest rank's time."""
    return flops_per_step * steps * world / (max_total_ms * 1e-3) / 1e12


def workload(config: int, tokens=None):
    """Workload `config`; with `tokens`, a dense prefill config regenerated at
    s_q = s_kv = tokens (same heads, list pattern and seed)."""
    import mla_inputs as mi
    if tokens is None:
        return mi.config(config)
    if config not in (1, 2, 3):
        raise SystemExit("--tokens applies to the dense prefill configs 1-3")
    h, pattern = (64, "recent") if config == 3 else (8, "causal")
    return mi.prefill_case(1000 + config, tokens, tokens, h, pattern=pattern,
                           name=f"c{config}_at_{tokens}_tokens")


def valid_entries(case) -> int:
    return int((case.indices >= 0).sum())


def step_flops(case) -> float:
    import mla_inputs as mi
    if hasattr(case, "kv_cache"):
        n_tok, h = case.batch * case.s_next, case.h_q
    else:
        n_tok, h = case.q.shape[0], case.q.shape[1]
    return mi.nominal_flops(n_tok, h, case.indices.shape[-1])


METRICS = {"fwd": "sparse-MLA fwd TFLOP/s at topk=2048 (nominal FLOPs)",
           "bwd": "sparse-MLA bwd TFLOP/s at topk=2048 (nominal FLOPs)",
           "causal": "indices-free causal MLA fwd TFLOP/s (every causal position)",
           "fp8": "sparse-MLA FP8-cache decode TFLOP/s at topk=2048 (nominal FLOPs)"}
MODE_SUFFIX = {"fwd": "", "bwd": " (backward: dq, dkv)", "causal": " (indices-free causal mode)",
               "fp8": ", FP8 cache (656-byte slots)"}


def attention_mode(args) -> str:
    fp8 = getattr(args, "fp8", False)
    if int(args.causal) + int(args.bwd) + int(fp8) > 1:
        raise SystemExit("--causal, --bwd and --fp8 are separate modes")
    return "causal" if args.causal else ("bwd" if args.bwd else ("fp8" if fp8 else "fwd"))


def check_mode(case, mode: str) -> None:
    if mode == "causal" and (hasattr(case, "kv_cache") or hasattr(case, "cu_seqlens_q")):
        raise SystemExit("--causal needs a dense prefill config (1-3)")
    if mode == "bwd" and hasattr(case, "kv_cache"):
        raise SystemExit("--bwd needs a prefill config (1-4)")
    if mode == "fp8" and not hasattr(case, "kv_cache"):
        raise SystemExit("--fp8 needs the paged decode config (5)")


def causal_entries(case) -> int:
    """Positions the indices-free causal mode attends to (queries are the last
    s_q of the s_kv positions)."""
    s_q, s_kv = case.q.shape[0], case.kv.shape[0]
    return sum(max(0, min(s_kv, t + s_kv - s_q + 1)) for t in range(s_q))


def mode_flops(case, mode: str) -> float:
    """FLOPs of one step: nominal 2 s_q h topk (576 + 512) for the forward,
    2 s_q h topk (3 576 + 2 512) for the backward (S recompute, dP, dQ, dK,
    dV), 2 h (576 + 512) per attended position for the causal mode."""
    if mode == "causal":
        return 2.0 * case.q.shape[1] * 1088 * causal_entries(case)
    if mode == "bwd":
        return 2.0 * case.q.shape[0] * case.q.shape[1] * case.indices.shape[-1] * (3 * 576 + 2 * 512)
    return step_flops(case)


def workload_name(case, config: int, tokens=None) -> str:
    if tokens is not None:
        return (f"{'wide-head' if config == 3 else 'dense'} prefill s_q=s_kv={tokens} h_q={case.q.shape[1]} "
                f"d_qk=576 d_v=512 topk=2048 bf16 (profiling size)")
    return _workload_name(config)


def _workload_name(config: int) -> str:
    names = {1: "tiny prefill s_q=s_kv=64 h_q=8",
             2: "mid prefill s_q=s_kv=2119 h_q=8",
             3: "wide-head prefill s_q=s_kv=8192 h_q=64",
             4: "packed varlen prefill 16384 tokens (8192,4096,2048,1024,1024) h_q=64",
             5: "paged decode batch=16 x 6 MTP tokens, contexts U[4096,32768], page 64, h_q=8"}
    return names[config] + " d_qk=576 d_v=512 topk=2048 bf16"


def h_q_of(case) -> int:
    return case.h_q if hasattr(case, "kv_cache") else case.q.shape[1]


def run_config(case, args, mode: str, world: int) -> dict:
    """The `config` object of both arms' lines (identical for the same
    workload and mode): the workload, its seed, the L2 rule of the GPU arm's
    timing and the parallelism."""
    return {"workload": workload_name(case, args.config, args.tokens) + MODE_SUFFIX[mode],
            "seed": 1000 + args.config,
            "l2": "256 MB buffer written before every timed step (cold L2)",
            "parallelism": f"replicas x{world}"}


# ----------------------------------------------------------------------------- oracle on host cores

def bwd_dout(case, config: int):
    """The upstream gradient both arms use for the backward: seeded N(0,1)
    rounded to bf16, shaped like the forward's output."""
    import torch
    g = torch.Generator().manual_seed(2000 + config)
    return torch.randn((case.q.shape[0], case.q.shape[1], 512), generator=g).to(torch.bfloat16)


def _oracle_worker_init(config: int, mode: str = "fwd"):
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    global _W_CASE, _W_MODE, _W_DOUT, _W_CACHE8
    _W_CASE = workload(config)
    _W_MODE = mode
    _W_DOUT = bwd_dout(_W_CASE, config) if mode == "bwd" else None
    if mode == "fp8":
        import mla_inputs as mi
        _W_CACHE8 = mi.quantize_fp8_slots(_W_CASE.kv_cache)


def _oracle_bwd_sample(orc, c, dout, tokens):
    """The oracle backward over a token sample: the sampled tokens' own
    gradients (dkv gets their contributions only)."""
    import torch
    if len(tokens) == 0:
        return
    sel = torch.tensor(list(tokens), dtype=torch.int64)
    if hasattr(c, "cu_seqlens_q"):
        cu = c.cu_seqlens_q.tolist()
        # the sample's sequences keep their order: count its tokens per sequence
        cu_s = [sum(1 for t in tokens if t < end) for end in cu]
        orc.sparse_mla_bwd_varlen(c.q[sel], c.kv, c.indices[sel], torch.tensor(cu_s, dtype=torch.int32),
                                  c.cu_seqlens_kv, c.sm_scale, dout[sel])
    else:
        orc.sparse_mla_bwd(c.q[sel], c.kv, c.indices[sel], c.sm_scale, dout[sel])


def _oracle_worker(tokens):
    from oracle import sparse_mla_oracle as orc
    c = _W_CASE
    t0 = time.perf_counter()
    if _W_MODE == "causal":
        orc.causal_mla_fwd(c.q, c.kv, c.sm_scale, tokens=tokens)
    elif _W_MODE == "bwd":
        _oracle_bwd_sample(orc, c, _W_DOUT, tokens)
    elif _W_MODE == "fp8":
        from oracle import fp8_kv_oracle as f8
        toks = [(t // c.s_next, t % c.s_next) for t in tokens]
        f8.sparse_mla_decode_fp8(c.q, _W_CACHE8, c.block_table, c.cache_seqlens, c.indices, c.sm_scale,
                                 c.page_size, tokens=toks)
    elif hasattr(c, "kv_cache"):
        toks = [(t // c.s_next, t % c.s_next) for t in tokens]
        orc.sparse_mla_decode(c.q, c.kv_cache, c.block_table, c.cache_seqlens, c.indices, c.sm_scale,
                              c.page_size, tokens=toks)
    elif hasattr(c, "cu_seqlens_q"):
        orc.sparse_mla_fwd_varlen(c.q, c.kv, c.indices, c.cu_seqlens_q, c.cu_seqlens_kv, c.sm_scale,
                                  tokens=tokens)
    else:
        orc.sparse_mla_fwd(c.q, c.kv, c.indices, c.sm_scale, tokens=tokens)
    return time.perf_counter() - t0


class OraclePool:
    """The oracle, unchanged, sharded by token over a spawn process pool with
    one single-threaded worker per host core.  mode: "fwd" (the forward of
    the workload's layout), "causal" (the indices-free causal forward) or
    "bwd" (the backward)."""

    def __init__(self, config: int, cores: int, mode: str = "fwd"):
        import multiprocessing as mp
        self.cores = cores
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(cores, initializer=_oracle_worker_init, initargs=(config, mode))
        self.pool.map(_oracle_worker, [[] for _ in range(cores)])   # wait for every worker

    def run(self, tokens):
        shards = [tokens[i::self.cores] for i in range(self.cores)]
        t0 = time.perf_counter()
        self.pool.map(_oracle_worker, shards)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_sample(case, config: int):
    """Token sample for one oracle step: the whole workload for configs 1, 2
    and 5; for the 8192/16384-token configs a seeded 1/16 sample."""
    import numpy as np
    n = case.batch * case.s_next if hasattr(case, "kv_cache") else case.q.shape[0]
    if config in (1, 2, 5):
        return list(range(n)), f"all {n} tokens of the workload"
    rng = np.random.default_rng(config)
    toks = sorted(rng.choice(n, n // 16, replace=False).tolist())
    return toks, f"seeded sample of {len(toks)} of {n} tokens (1/16), scaled by FLOPs"


# ----------------------------------------------------------------------------- arms

def indexer_config(args, world: int) -> dict:
    """The `config` object of both arms' indexer lines (identical)."""
    name = {1: "tiny prefill s_q=s_kv=64", 2: "mid prefill s_q=s_kv=2119", 3: "prefill s_q=s_kv=8192",
            4: "packed varlen prefill 16384 tokens (8192,4096,2048,1024,1024)",
            5: "paged decode 16 requests x 6 MTP rows, contexts U[4096,32768], page 64"}[args.config]
    return {"workload": f"DSA indexer {name} h_idx=64 d_idx=128 topk=2048 (lists for the sparse-MLA "
                        f"forward; one logits chunk)", "seed": 1000 + args.config,
            "l2": "256 MB buffer written before every timed step (cold L2)",
            "parallelism": f"replicas x{world}"}


def run_reference_indexer(args, world=1):
    case = indexer_workload(args.config)
    info = indexer_rows(case)
    flops, _, scored_pos, _ = indexer_costs(case, info)
    cores = os.cpu_count() or 1
    pool = IndexerOraclePool(args.config, cores)
    rows, sample = indexer_oracle_sample(info, args.config)
    part = sum(info[r][0] for r in rows) / max(1, scored_pos)
    for _ in range(args.warmup):
        pool.run(rows)
    times = [pool.run(rows) for _ in range(args.steps)]
    pool.close()
    total = sum(times)
    value = flops * part * args.steps / total / 1e12
    line = {
        "impl": "reference",
        "metric": "DSA indexer scores + top-k TFLOP/s at topk=2048 (2*h_idx*d_idx per scored position)",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": indexer_config(args, world),
        "timing": "host wall clock of the oracle over the sample on the host cores (no L2 flush applies)",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    if args.indexer:
        return run_reference_indexer(args, world)
    if args.tokens is not None:
        raise SystemExit("--tokens is a profiling size for the CUDA arm only")
    mode = attention_mode(args)
    case = workload(args.config)
    check_mode(case, mode)
    cores = os.cpu_count() or 1
    pool = OraclePool(args.config, cores, mode)
    toks, sample = oracle_sample(case, args.config)
    n_tok = case.batch * case.s_next if hasattr(case, "kv_cache") else case.q.shape[0]
    flops = mode_flops(case, mode) * len(toks) / n_tok
    for _ in range(args.warmup):
        pool.run(toks)
    times = [pool.run(toks) for _ in range(args.steps)]
    pool.close()
    total = sum(times)
    value = flops * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRICS[mode],
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": run_config(case, args, mode, world),
        "timing": "host wall clock of the oracle over the sample on the host cores (no L2 flush applies)",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def fwd_runner(smla, case, dev, stream):
    """Device-resident inputs of one forward workload and a closure that runs
    its forward once (dense, packed or paged, as the workload's layout is);
    returns (closure, launches per call, device tensors to free)."""
    d = lambda t: t.to(dev)
    if hasattr(case, "kv_cache"):
        inp = dict(q=d(case.q), kv=d(case.kv_cache), bt=d(case.block_table), sl=d(case.cache_seqlens),
                   idx=d(case.indices))
        need = smla.decode_workspace_size(case.batch, case.s_next, case.h_q, case.indices.shape[-1])
        ws = torch_empty_bytes(max(1, need), dev)
        out = torch_empty_out((case.batch, case.s_next, case.h_q), dev)

        def call():
            smla.sparse_mla_decode(inp["q"], inp["kv"], inp["bt"], inp["sl"], inp["idx"], case.sm_scale,
                                   case.page_size, workspace=ws, out=out[0], lse=out[1], stream=stream)
        return call, 1, [inp, ws, out]
    inp = dict(q=d(case.q), kv=d(case.kv), idx=d(case.indices))
    out = torch_empty_out((case.q.shape[0], case.q.shape[1]), dev)
    if hasattr(case, "cu_seqlens_q"):
        inp.update(cuq=d(case.cu_seqlens_q), cuk=d(case.cu_seqlens_kv))

        def call():
            smla.sparse_mla_fwd_varlen(inp["q"], inp["kv"], inp["idx"], inp["cuq"], inp["cuk"], case.sm_scale,
                                       out=out[0], lse=out[1], stream=stream)
    else:
        def call():
            smla.sparse_mla_fwd(inp["q"], inp["kv"], inp["idx"], case.sm_scale, out=out[0], lse=out[1],
                                stream=stream)
    return call, 1, [inp, out]


def torch_empty_bytes(n, dev):
    import torch
    return torch.empty(n, dtype=torch.uint8, device=dev)


def torch_empty_out(lead, dev):
    """(out [*lead, 512] bf16, lse [*lead] fp32) on dev."""
    import torch
    return (torch.empty((*lead, 512), dtype=torch.bfloat16, device=dev),
            torch.empty(lead, dtype=torch.float32, device=dev))


FP8_SLOT_BYTES = 656


def fp8_runner(smla, case, dev, stream):
    """The paged-decode workload with its cache written as FP8 slots (the
    656-byte layout of sparse_mla_decode_fp8): device inputs and a closure
    that runs one FP8 decode."""
    import mla_inputs as mi
    d = lambda t: t.to(dev)
    inp = dict(q=d(case.q), kv=d(mi.quantize_fp8_slots(case.kv_cache)), bt=d(case.block_table),
               sl=d(case.cache_seqlens), idx=d(case.indices))
    need = smla.decode_workspace_size(case.batch, case.s_next, case.h_q, case.indices.shape[-1])
    ws = torch_empty_bytes(max(1, need), dev)
    out = torch_empty_out((case.batch, case.s_next, case.h_q), dev)

    def call():
        smla.sparse_mla_decode_fp8(inp["q"], inp["kv"], inp["bt"], inp["sl"], inp["idx"], case.sm_scale,
                                   case.page_size, workspace=ws, out=out[0], lse=out[1], stream=stream)
    return call, 1, [inp, ws, out]


PAGES_TRIALS = 5    # the pages' timing: interleaved trials ...
PAGES_CALLS = 20    # ... each the median of this many warm calls
PAGES_LEAD_CYCLES = 4_000_000   # ~2 ms of device-side wait ahead of a trial's timed calls


def config_records(smla, dev, stream, steps: int, warmup: int, flush, peaks) -> dict:
    """Per-workload forward records for all five workloads: the time per call
    with a cold L2 (mean over `steps` calls, CUDA events on the launching
    stream, a 256 MB buffer written before each) and with a warm L2 (median),
    the per-shape roofline (max of the nominal-FLOP term at the measured bf16
    peak and the valid gathered-KV bytes at the measured HBM copy bandwidth),
    the fraction of it reached, the tensor-only fraction (FLOP term / time),
    and the profiled DRAM traffic of the launch when the committed ncu summary
    matches the current kernel sources.  Then the pages' own timing of each
    workload: PAGES_TRIALS trials with the workloads rotated between them,
    each the median of PAGES_CALLS warm-L2 calls after 3 warm-up calls, and
    the median of the trial medians (no L2 flush, as on the pages)."""
    import torch
    p_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    p_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    recs = {}
    alive = {}   # workload -> (closure, device tensors), for the interleaved trials
    for c in (1, 2, 3, 4, 5, "5_fp8"):
        fp8 = c == "5_fp8"
        case = workload(5 if fp8 else c)
        call, launches, keep = (fp8_runner if fp8 else fwd_runner)(smla, case, dev, stream)
        row_bytes = FP8_SLOT_BYTES if fp8 else KV_ROW_BYTES
        for _ in range(max(3, warmup)):
            call()
        torch.cuda.synchronize(dev)
        cold, warm = [], []
        for i in range(2 * steps):
            if i < steps:
                flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            (cold if i < steps else warm).append((a, b))
        torch.cuda.synchronize(dev)
        us = statistics.mean(a.elapsed_time(b) for a, b in cold) * 1e3
        us_warm = statistics.median(a.elapsed_time(b) for a, b in warm) * 1e3
        valid = valid_entries(case)
        flops = step_flops(case)
        t_flop = flops / (p_tf * 1e12) * 1e6
        t_byte = valid * row_bytes / (p_bw * 1e9) * 1e6
        roof = max(t_flop, t_byte)
        recs[str(c)] = {
            "workload": (_workload_name(5) + ", FP8 cache (656-byte slots)") if fp8 else _workload_name(c),
            "us_per_call": us, "us_per_call_warm_l2": us_warm,
            "roofline_us": roof, "bound": "hbm" if t_byte >= t_flop else "tensor",
            "roofline_frac": roof / us, "tensor_only_frac": t_flop / us,
            "tflops": flops / (us * 1e-6) / 1e12, "gathered_kv_GBps": valid * row_bytes / (us * 1e-6) / 1e9,
            "gathered_row_bytes": row_bytes,
            "valid_entries": valid, "nominal_flops": flops, "launches_per_call": launches,
            "traffic": profiled_traffic(c, "fwd"),
        }
        alive[str(c)] = (call, keep, roof, flops, valid * row_bytes)
        del keep, call
    trials = {c: [] for c in alive}
    for _ in range(PAGES_TRIALS):
        for c, (call, _, _, _, _) in alive.items():
            for _ in range(3):
                call()
            # a device-side wait first, so that the host has queued all the
            # timed calls before the first runs: the events then time the
            # GPU, not the host's launch gaps (the L2 stays warm)
            if hasattr(torch.cuda, "_sleep"):
                torch.cuda._sleep(PAGES_LEAD_CYCLES)
            evs = []
            for _ in range(PAGES_CALLS):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                call()
                b.record(stream)
                evs.append((a, b))
            torch.cuda.synchronize(dev)
            trials[c].append(statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3)
    for c, (_, _, roof, flops, nbytes) in alive.items():
        us_p = statistics.median(trials[c])
        recs[c]["pages_method"] = {
            "us_per_call": us_p, "trial_medians_us": trials[c], "roofline_frac": roof / us_p,
            "tflops": flops / (us_p * 1e-6) / 1e12, "gathered_kv_GBps": nbytes / (us_p * 1e-6) / 1e9,
            "method": f"{PAGES_TRIALS} trials, workloads rotated between trials, each the median of {PAGES_CALLS} "
                      "warm-L2 calls after 3 warm-up calls, queued behind a device-side wait so that the events "
                      "time the GPU; median of the trial medians (no L2 flush)"}
    alive.clear()
    torch.cuda.empty_cache()
    return recs


def run_ours(args, rank, world, dist):
    import torch
    import serving_sparse_mla_gb300 as smla

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = smla.load()   # raises if the CUDA library is missing: no fallback

    # The oracle pool (spawn) starts before the first GPU work.
    pool = None
    if rank == 0 and not args.no_cpu_baseline and args.tokens is None:
        pool = OraclePool(args.config, os.cpu_count() or 1, attention_mode(args))

    case = workload(args.config, args.tokens)
    stream = torch.cuda.current_stream(dev)
    is_decode = hasattr(case, "kv_cache")
    is_varlen = hasattr(case, "cu_seqlens_q")
    mode = attention_mode(args)
    check_mode(case, mode)
    n_tok = case.batch * case.s_next if is_decode else case.q.shape[0]
    flops = mode_flops(case, mode)
    valid = causal_entries(case) if args.causal else valid_entries(case)
    # The HBM roofline counts the gathered KV rows; the backward's fp32 dkv
    # reductions (576 x 4 B per valid entry and 32-head unit, L2-resident
    # red.global.add) are reported beside it, not as HBM bytes.
    kv_bytes = valid * (FP8_SLOT_BYTES if mode == "fp8" else KV_ROW_BYTES)
    red_bytes = valid * 2304 * (2 if h_q_of(case) > 16 else 1) if args.bwd else 0

    # device-resident inputs
    d = lambda t: t.to(dev)
    if is_decode:
        kv_in = case.kv_cache
        if mode == "fp8":
            import mla_inputs as mi
            kv_in = mi.quantize_fp8_slots(case.kv_cache)
        inputs = dict(q=d(case.q), kv=d(kv_in), bt=d(case.block_table), sl=d(case.cache_seqlens),
                      idx=d(case.indices))
        ws = torch.empty(max(1, smla.decode_workspace_size(case.batch, case.s_next, case.h_q, 2048)),
                         dtype=torch.uint8, device=dev)
    elif is_varlen and args.bwd:
        inputs = dict(q=d(case.q), kv=d(case.kv), idx=d(case.indices), cuq=d(case.cu_seqlens_q),
                      cuk=d(case.cu_seqlens_kv))
        o_fwd, l_fwd = smla.sparse_mla_fwd_varlen(inputs["q"], inputs["kv"], inputs["idx"], inputs["cuq"],
                                                  inputs["cuk"], case.sm_scale)
        inputs.update(out=o_fwd, lse=l_fwd, dout=bwd_dout(case, args.config).to(dev))
        dq_buf = torch.empty(case.q.shape, dtype=torch.float32, device=dev)
        dkv_buf = torch.empty((case.kv.shape[0], 576), dtype=torch.float32, device=dev)
    elif is_varlen:
        inputs = dict(q=d(case.q), kv=d(case.kv), idx=d(case.indices), cuq=d(case.cu_seqlens_q),
                      cuk=d(case.cu_seqlens_kv))
    elif args.causal:
        inputs = dict(q=d(case.q), kv=d(case.kv))
    elif args.bwd:
        inputs = dict(q=d(case.q), kv=d(case.kv), idx=d(case.indices))
        o_fwd, l_fwd = smla.sparse_mla_fwd(inputs["q"], inputs["kv"], inputs["idx"], case.sm_scale)
        inputs.update(out=o_fwd, lse=l_fwd, dout=bwd_dout(case, args.config).to(dev))
        dq_buf = torch.empty(case.q.shape, dtype=torch.float32, device=dev)
        dkv_buf = torch.empty((case.kv.shape[0], 576), dtype=torch.float32, device=dev)
    else:
        inputs = dict(q=d(case.q), kv=d(case.kv), idx=d(case.indices))
    h_q = case.h_q if is_decode else case.q.shape[1]
    out = torch.empty((n_tok, h_q, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((n_tok, h_q), dtype=torch.float32, device=dev)

    def call(inp):
        if is_decode and mode == "fp8":
            smla.sparse_mla_decode_fp8(inp["q"], inp["kv"], inp["bt"], inp["sl"], inp["idx"], case.sm_scale,
                                       case.page_size, workspace=ws, out=out.view(case.batch, case.s_next, h_q, 512),
                                       lse=lse.view(case.batch, case.s_next, h_q), stream=stream)
        elif is_decode:
            smla.sparse_mla_decode(inp["q"], inp["kv"], inp["bt"], inp["sl"], inp["idx"], case.sm_scale,
                                   case.page_size, workspace=ws, out=out.view(case.batch, case.s_next, h_q, 512),
                                   lse=lse.view(case.batch, case.s_next, h_q), stream=stream)
        elif is_varlen and args.bwd:
            smla.sparse_mla_bwd_varlen(inp["q"], inp["kv"], inp["idx"], inp["cuq"], inp["cuk"], case.sm_scale,
                                       inp["out"], inp["lse"], inp["dout"], dq=dq_buf, dkv=dkv_buf, stream=stream)
        elif is_varlen:
            smla.sparse_mla_fwd_varlen(inp["q"], inp["kv"], inp["idx"], inp["cuq"], inp["cuk"], case.sm_scale,
                                       out=out, lse=lse, stream=stream)
        elif args.causal:
            smla.sparse_mla_fwd_causal(inp["q"], inp["kv"], case.sm_scale, out=out, lse=lse, stream=stream)
        elif args.bwd:
            smla.sparse_mla_bwd(inp["q"], inp["kv"], inp["idx"], case.sm_scale, inp["out"], inp["lse"], inp["dout"],
                                dq=dq_buf, dkv=dkv_buf, stream=stream)
        else:
            smla.sparse_mla_fwd(inp["q"], inp["kv"], inp["idx"], case.sm_scale, out=out, lse=lse, stream=stream)

    # One kernel of ours per call (the decode's split merge runs inside the
    # forward; the counter memset before it is a runtime memset node).
    launches_per_step = 1
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    def timed_loop(k, body, flush_l2=True):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
        for i in range(k):
            if flush_l2:
                flush.zero_()
            starts[i].record(stream)
            body()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    for _ in range(max(3, args.warmup)):
        call(inputs)
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local, args.clock_log or tempfile.gettempdir())
    nvml = NvmlClockSampler(dev)
    sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    nvml.start()
    times = timed_loop(args.steps, lambda: call(inputs))
    torch.cuda.synchronize(dev)
    nvml_clocks = nvml.stop()
    barrier()
    smi_clocks = sampler.stop()
    clocks = nvml_clocks or smi_clocks
    # secondary: warm L2 (the pages' method has no flush)
    warm = timed_loop(max(args.steps, 20), lambda: call(inputs), flush_l2=False)

    # end to end through the C ABI with host buffers: pinned H2D of the inputs,
    # the call, D2H of its results (out and lse; dq and dkv for the backward),
    # all inside the timed region
    host = {k: v.cpu().pin_memory() for k, v in inputs.items()}
    dev2 = {k: torch.empty_like(v) for k, v in inputs.items()}
    results = [dq_buf, dkv_buf] if args.bwd else [out, lse]
    res_h = [torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in results]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(r.numel() * r.element_size() for r in results)

    def e2e_step():
        for k in host:
            dev2[k].copy_(host[k], non_blocking=True)
        call(dev2)
        for rh, r in zip(res_h, results):
            rh.copy_(r, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e2e_times = timed_loop(args.steps, e2e_step)
    barrier()

    total_ms, e2e_ms = max_over_ranks([sum(times), sum(e2e_times)], dist, dev)

    if rank != 0:
        return 0

    peaks, peak_kind = load_peaks()
    ms = total_ms / args.steps
    us = ms * 1e3
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    p_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    p_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    roof_us = max(flops / (p_tf * 1e12), kv_bytes / (p_bw * 1e9)) * 1e6
    bound = "hbm" if kv_bytes / (p_bw * 1e9) >= flops / (p_tf * 1e12) else "tensor"
    fwd_ms = ms  # one forward launch per step (the decode merges its split units inside it)
    if bound == "hbm":
        achieved = kv_bytes / (fwd_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": p_bw, "unit": "GB/s",
                    "frac": achieved / p_bw, "traffic": None if args.causal else profiled_traffic("5_fp8" if mode == "fp8" else args.config,
                                                                                "bwd" if args.bwd else "fwd"),
                    "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                    "algorithmic_bytes_per_launch": kv_bytes,
                    "note": f"achieved = valid entries x {kv_bytes // max(1, valid)} B gathered / mean launch time "
                            "(cold L2)"}
    else:
        achieved = flops / (fwd_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": p_tf, "unit": "TFLOP/s",
                    "frac": achieved / p_tf, "traffic": None if args.causal else profiled_traffic(args.config, "bwd" if args.bwd else "fwd"),
                    "peak_kind": f"{peak_kind} bf16 (burst)", "algorithmic_flops_per_launch": flops}

    cpu = None
    if pool is not None:
        toks, sample = oracle_sample(case, args.config)
        wall = pool.run(toks)
        cpu = {"value": flops * len(toks) / n_tok / wall / 1e12, "unit": "TFLOP/s", "cores": pool.cores,
               "kind": "oracle", "sample": sample, "seconds": wall}
        pool.close()

    line = {
        "metric": METRICS[mode],
        "value": whole_job_tflops(flops, args.steps, world, total_ms), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": run_config(case, args, mode, world),
        "us_per_call": us, "tflops_per_gpu": tflops, "gathered_kv_GBps": gbs,
        "roofline_us": roof_us, "roofline_pct": 100.0 * roof_us / us,
        "warm_l2": {"us_per_call": statistics.median(warm) * 1e3,
                    "roofline_pct": 100.0 * roof_us / (statistics.median(warm) * 1e3)},
        "valid_entries": valid, "nominal_flops": flops,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": flops * world / (e2e_ms / args.steps * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if args.bwd:
        line["dkv_reduction"] = {
            "bytes_per_launch": red_bytes, "GBps": red_bytes / (ms * 1e-3) / 1e9,
            "note": "fp32 red.global.add of dK/dV rows into dkv (576 x 4 B per valid entry and 32-head unit); "
                    "the rows stay in L2, so this is L2 traffic, not counted in the HBM roofline and not "
                    "divided by any measured peak"}
    if mode == "fwd" and args.tokens is None and not args.no_all_configs:
        line["configs"] = config_records(smla, dev, stream, args.steps, args.warmup, flush, peaks)
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- DSA indexer

IDX_TOPK = 2048


def indexer_workload(config: int):
    """The indexer inputs on the token shape of workload `config`."""
    import mla_inputs as mi
    seed = 1000 + config
    if config == 1:
        return mi.indexer_case(seed, 64, 64)
    if config == 2:
        return mi.indexer_case(seed, 2119, 2119)
    if config == 3:
        return mi.indexer_case(seed, 8192, 8192)
    if config == 4:
        return mi.indexer_varlen_case(seed, mi.VARLEN_C4, mi.VARLEN_C4)
    # decode: 16 requests x 6 MTP rows over a paged key cache, contexts U[4096, 32768]
    return mi.indexer_paged_case(seed, 16, 6, 4096, 32768)


def indexer_rows(case):
    """Per query row: (visible length, scored?)."""
    if hasattr(case, "k_cache"):
        s_next = case.q_idx.shape[1]
        out = []
        for lk in case.cache_seqlens.tolist():
            for t in range(s_next):
                v = max(0, min(lk, t + lk - s_next + 1))
                out.append((v, v > case.topk))
        return out
    s_q, s_kv = case.q_idx.shape[0], case.k_idx.shape[0]
    if case.cu_seqlens_q is None:
        seqs = [(0, s_q, s_kv)]
    else:
        cq, ck = case.cu_seqlens_q.tolist(), case.cu_seqlens_kv.tolist()
        seqs = [(cq[b], cq[b + 1] - cq[b], ck[b + 1] - ck[b]) for b in range(len(cq) - 1)]
    out = []
    for _, lq, lk in seqs:
        for t in range(lq):
            v = max(0, min(lk, t + lk - lq + 1))
            out.append((v, v > case.topk))
    return out


def _idx_oracle_init(config: int):
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    global _W_IDX
    _W_IDX = indexer_workload(config)


def _idx_oracle_worker(rows):
    from oracle import dsa_indexer_oracle as ido
    c = _W_IDX
    t0 = time.perf_counter()
    if rows and hasattr(c, "k_cache"):
        ido.dsa_indices_paged(c.q_idx, c.k_cache, c.weights, c.block_table, c.cache_seqlens, c.topk, c.page,
                              rows=rows)
    elif rows:
        if c.cu_seqlens_q is None:
            ido.dsa_indices(c.q_idx, c.k_idx, c.weights, c.topk, rows=rows)
        else:
            ido.dsa_indices_varlen(c.q_idx, c.k_idx, c.weights, c.cu_seqlens_q, c.cu_seqlens_kv, c.topk, rows=rows)
    return time.perf_counter() - t0


class IndexerOraclePool(OraclePool):
    """The indexer oracle, unchanged, sharded by query row over a spawn pool
    of single-threaded workers (one per host core)."""

    def __init__(self, config: int, cores: int):
        import multiprocessing as mp
        self.cores = cores
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(cores, initializer=_idx_oracle_init, initargs=(config,))
        self.pool.map(_idx_oracle_worker, [[] for _ in range(cores)])

    def run(self, rows):
        shards = [rows[i::self.cores] for i in range(self.cores)]
        t0 = time.perf_counter()
        self.pool.map(_idx_oracle_worker, shards)
        return time.perf_counter() - t0


def indexer_oracle_sample(rows_info, config: int):
    """Rows for one oracle step: every scored row of the workload (the
    oracle's own cost; rows that see at most topk positions need no score).
    At 8192 tokens that is ~25 s of single-core work."""
    scored = [i for i, (_, sc) in enumerate(rows_info) if sc]
    return scored, f"all {len(scored)} scored rows of the workload"


def indexer_costs(case, rows_info):
    """Algorithmic FLOPs and bytes of one indexer step: the score contraction
    over scored (row, position) pairs, and the HBM bytes of Q, K and the
    weights of scored rows, the logits written and read back once, and the
    lists written."""
    h, d = case.q_idx.shape[-2], case.q_idx.shape[-1]
    scored_pos = sum(v for v, sc in rows_info if sc)
    scored_rows = sum(1 for _, sc in rows_info if sc)
    flops = 2.0 * h * d * scored_pos
    n_keys = int(case.cache_seqlens.sum()) if hasattr(case, "k_cache") else case.k_idx.shape[0]
    byts = (scored_rows * h * (d * 2 + 4) + n_keys * d * 2 + scored_pos * 4 * 2
            + len(rows_info) * case.topk * 4)
    return flops, byts, scored_pos, scored_rows


def run_indexer(args, rank, world, dist):
    import torch
    import serving_sparse_mla_gb300 as smla

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    smla.load()   # raises if the CUDA library is missing: no fallback
    pool = None
    if rank == 0 and not args.no_cpu_baseline:
        pool = IndexerOraclePool(args.config, os.cpu_count() or 1)

    case = indexer_workload(args.config)
    info = indexer_rows(case)
    flops, byts, scored_pos, scored_rows = indexer_costs(case, info)
    paged = hasattr(case, "k_cache")
    stream = torch.cuda.current_stream(dev)
    if paged:
        total_q = case.q_idx.shape[0] * case.q_idx.shape[1]
        total_kv = int(case.cache_seqlens.sum())
        longest = int(case.cache_seqlens.max())
        inputs = {"q": case.q_idx.to(dev), "k": case.k_cache.to(dev), "w": case.weights.to(dev),
                  "bt": case.block_table.to(dev), "sl": case.cache_seqlens.to(dev)}
    else:
        total_q, total_kv = case.q_idx.shape[0], case.k_idx.shape[0]
        longest = case.max_seqlen_kv
        inputs = {"q": case.q_idx.to(dev), "k": case.k_idx.to(dev), "w": case.weights.to(dev)}
        if case.cu_seqlens_q is not None:
            inputs.update(cq=case.cu_seqlens_q.to(dev), ck=case.cu_seqlens_kv.to(dev))
    need = smla.dsa_indexer_workspace_size(total_q, longest, case.topk)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)     # one chunk: every row's logits
    idx = torch.empty((total_q, case.topk), dtype=torch.int32, device=dev)
    stride = (longest + 3) // 4 * 4
    logits = ws[:max(need, 16)].view(torch.float32)[:max(need, 16) // 4]
    first = 0 if paged or case.cu_seqlens_q is not None else max(0, min(total_q, case.topk - (total_kv - total_q)))

    def call(inp):
        if paged:
            smla.dsa_indexer_topk_paged(inp["q"], inp["k"], inp["w"], inp["bt"], inp["sl"], case.topk, longest,
                                        workspace=ws, indices=idx.view(inp["q"].shape[0], -1, case.topk),
                                        stream=stream)
        else:
            smla.dsa_indexer_topk(inp["q"], inp["k"], inp["w"], case.topk, inp.get("cq"), inp.get("ck"), longest,
                                  workspace=ws, indices=idx, stream=stream)

    def scores_only(inp):
        # the launch dsa_indexer_topk makes for the scores of its one chunk
        view = logits[:(total_q - first) * stride].view(total_q - first, stride)
        if paged:
            smla.dsa_indexer_scores_paged(inp["q"], inp["k"], inp["w"], inp["bt"], inp["sl"], longest, row0=0,
                                          n_rows=total_q, skip_len=case.topk, scores=view, stream=stream)
        else:
            smla.dsa_indexer_scores(inp["q"], inp["k"], inp["w"], inp.get("cq"), inp.get("ck"), row0=first,
                                    n_rows=total_q - first, skip_len=case.topk, scores=view,
                                    max_seqlen_kv=longest, stream=stream)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def timed_loop(k, body, flush_l2=True):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
        for i in range(k):
            if flush_l2:
                flush.zero_()
            starts[i].record(stream)
            body()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in zip(starts, ends)]

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        call(inputs)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local, args.clock_log or tempfile.gettempdir())
    nvml = NvmlClockSampler(dev)
    sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    nvml.start()
    times = timed_loop(args.steps, lambda: call(inputs))
    torch.cuda.synchronize(dev)
    nvml_clocks = nvml.stop()
    barrier()
    smi_clocks = sampler.stop()
    clocks = nvml_clocks or smi_clocks
    # the dominant kernel alone (scores), same launch, for the roofline
    sc_times = timed_loop(args.steps, lambda: scores_only(inputs)) if scored_rows else []

    host = {k: v.cpu().pin_memory() for k, v in inputs.items()}
    dev2 = {k: torch.empty_like(v) for k, v in inputs.items()}
    res_h = torch.empty(idx.shape, dtype=idx.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = idx.numel() * idx.element_size()

    def e2e_step():
        for k in host:
            dev2[k].copy_(host[k], non_blocking=True)
        call(dev2)
        res_h.copy_(idx, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e2e_times = timed_loop(args.steps, e2e_step)
    barrier()
    total_ms, e2e_ms = max_over_ranks([sum(times), sum(e2e_times)], dist, dev)
    if rank != 0:
        return 0

    peaks, peak_kind = load_peaks()
    p_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    p_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ms = total_ms / args.steps
    roof_us = max(flops / (p_tf * 1e12), byts / (p_bw * 1e9)) * 1e6
    roofline = None
    if sc_times:
        sc_ms = statistics.mean(sc_times)
        sc_flops = flops
        sc_bytes = scored_rows * case.q_idx.shape[-2] * (case.q_idx.shape[-1] * 2 + 4) + total_kv * 256 + scored_pos * 4
        if sc_flops / (p_tf * 1e12) >= sc_bytes / (p_bw * 1e9):
            ach = sc_flops / (sc_ms * 1e-3) / 1e12
            roofline = {"bound": "tensor", "achieved": ach, "peak": p_tf, "unit": "TFLOP/s", "frac": ach / p_tf,
                        "traffic": profiled_traffic(args.config, "idx"), "kernel": "dsa_scores_kernel", "peak_kind": f"{peak_kind} bf16 (burst)",
                        "algorithmic_flops_per_launch": sc_flops, "us_per_launch": sc_ms * 1e3}
        else:
            ach = sc_bytes / (sc_ms * 1e-3) / 1e9
            roofline = {"bound": "hbm", "achieved": ach, "peak": p_bw, "unit": "GB/s", "frac": ach / p_bw,
                        "traffic": profiled_traffic(args.config, "idx"), "kernel": "dsa_scores_kernel", "peak_kind": f"{peak_kind} copy bandwidth",
                        "algorithmic_bytes_per_launch": sc_bytes, "us_per_launch": sc_ms * 1e3}
    cpu = None
    if pool is not None:
        rows, sample = indexer_oracle_sample(info, args.config)
        wall = pool.run(rows)
        part = sum(info[r][0] for r in rows) / max(1, scored_pos)
        cpu = {"value": flops * part / wall / 1e12 if rows else None, "unit": "TFLOP/s", "cores": pool.cores,
               "kind": "oracle", "sample": sample, "seconds": wall}
        pool.close()
    launches = 2 if scored_rows else 1
    line = {
        "metric": "DSA indexer scores + top-k TFLOP/s at topk=2048 (2*h_idx*d_idx per scored position)",
        "value": whole_job_tflops(flops, args.steps, world, total_ms), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": indexer_config(args, world),
        "us_per_call": ms * 1e3, "roofline_us": roof_us, "roofline_pct": 100.0 * roof_us / (ms * 1e3),
        "scored_rows": scored_rows, "scored_positions": scored_pos, "algorithmic_bytes": byts,
        "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": flops * world / (e2e_ms / args.steps * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        tdist.init_process_group(backend=backend)
        dist = tdist
    try:
        if args.indexer:
            return run_indexer(args, rank, world, dist)
        return run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
