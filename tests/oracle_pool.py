"""Whole-workload parity on the host cores: the float64 oracle over token
shards in a spawn process pool (one single-threaded worker per core), each
worker comparing its shard of the CUDA outputs with the oracle's and sending
back only statistics.  Test infrastructure: it imports the oracle, and only
tests use it.

The pool is started with the "spawn" method, so it is safe after the CUDA
context exists (a forked child of a CUDA process can hang).  Nothing crosses
the process boundary as a torch tensor: the KV rows (bf16 bits, or the FP8
cache's bytes) are written once to a temporary .npy file that every worker
memory-maps read-only, and each shard's q, index rows and CUDA results go as
numpy arrays.
"""
from __future__ import annotations

import os
import shutil
import tempfile
from typing import Dict, List

import numpy as np

_W: Dict = {}
_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of bf16 numbers given as their uint16 bits."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bits(t) -> np.ndarray:
    """uint16 bits of a bf16 CPU tensor."""
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _init(layout: str, kv_path: str, sm_scale: float, extra: dict):
    _W.update(layout=layout, kv=np.load(kv_path, mmap_mode="r"), sm_scale=sm_scale, extra=extra)


def _gather(r):
    """Rows r of the KV rows as float64 or, for the FP8 layout, the cache
    slots dequantized by the oracle."""
    sel = np.asarray(_W["kv"][r])
    if _W["layout"] == "paged_fp8":
        from oracle import fp8_kv_oracle as f8
        return f8.dequantize_slots(sel)
    return bf16_bits_to_f64(sel)


def _rows(layout, extra, t, idx_t, kv_rows):
    from oracle import sparse_mla_oracle as orc
    if layout == "dense":
        return orc.rows_dense(idx_t, kv_rows)
    if layout == "varlen":
        cu_q, cu_k = extra["cu_q"], extra["cu_k"]
        b = int(np.searchsorted(cu_q, t, side="right") - 1)
        return orc.rows_varlen(idx_t, int(cu_k[b]), int(cu_k[b + 1] - cu_k[b]))
    b = t // extra["s_next"]   # "paged" and "paged_fp8"
    return orc.rows_paged(idx_t, extra["table"][b], int(extra["lens"][b]), extra["page"], extra["num_blocks"])


def _shard(payload):
    """Compare one shard.  payload: tokens (global ids), q bits [n, h, 576]
    uint16, idx [n, topk] int64, gpu_out [n, h, 512] float32, gpu_lse [n, h]."""
    from oracle import sparse_mla_oracle as orc
    from tests.parity import compare, fp8_rounding_sigma, pv_rounding_sigma, tight_ratio
    sigma_of = fp8_rounding_sigma if _W["layout"] == "paged_fp8" else pv_rounding_sigma
    toks, q_bits, idx, g_out, g_lse = payload
    kv_rows = _W["kv"].shape[0]
    res = {"n": 0, "max_dout": 0.0, "max_dlse": 0.0, "tight": 0.0, "tight_full": 0.0, "fail": None}
    for i, t in enumerate(toks):
        r = _rows(_W["layout"], _W["extra"], int(t), idx[i], kv_rows)
        K = _gather(r)
        qt = bf16_bits_to_f64(q_bits[i])
        ro, rl = orc.attend(qt, K, _W["sm_scale"], 512)
        try:
            do, dl = compare(g_out[i:i + 1], g_lse[i:i + 1], ro[None], rl[None], f"token {t}")
        except AssertionError as e:   # report the first failure, keep the statistics going
            if res["fail"] is None:
                res["fail"] = str(e)
            continue
        res["max_dout"] = max(res["max_dout"], do)
        res["max_dlse"] = max(res["max_dlse"], dl)
        if r.size:
            tr = tight_ratio(g_out[i], ro, sigma_of(qt, K, _W["sm_scale"]))
            res["tight"] = max(res["tight"], tr)
            if r.size == idx.shape[1]:
                res["tight_full"] = max(res["tight_full"], tr)
        res["n"] += 1
    return res


def check_all_tokens(layout: str, q, kv, indices, gpu_out, gpu_lse, sm_scale: float, extra=None,
                     cores: int = 0, shard_tokens: int = 64) -> dict:
    """Every token of a workload against the oracle.  q [n, h, 576] bf16 CPU,
    indices [n, topk] int32 CPU, gpu_out [n, h, 512] and gpu_lse [n, h] (CPU
    tensors, the CUDA results).  layout and kv: "dense" or "varlen" (extra:
    cu_q, cu_k) with kv the bf16 rows [rows, 576]; "paged" (extra: table,
    lens, page, num_blocks, s_next) with kv the bf16 cache as [slots, 576];
    "paged_fp8" as "paged", kv the FP8 cache as uint8 [slots, 656].  Returns
    the worst |dout|, |dlse|, tight-check ratios (all tokens and full-list
    tokens) and the first failure message, if any."""
    import multiprocessing as mp
    import torch
    extra = {k: (v.numpy().astype(np.int64) if isinstance(v, torch.Tensor) else v)
             for k, v in (extra or {}).items()}
    n = q.shape[0]
    idx = indices.reshape(n, -1).numpy().astype(np.int64)
    kv_np = kv.contiguous().numpy() if kv.dtype == torch.uint8 else _bits(kv)
    q_bits = _bits(q)
    cores = cores or (os.cpu_count() or 1)
    payloads: List = []
    for a in range(0, n, shard_tokens):
        b = min(n, a + shard_tokens)
        payloads.append((np.arange(a, b), q_bits[a:b].copy(), idx[a:b], gpu_out[a:b].float().numpy(),
                         gpu_lse[a:b].float().numpy()))
    tmp = tempfile.mkdtemp(prefix="oracle_pool_")
    kv_path = os.path.join(tmp, "kv.npy")
    np.save(kv_path, kv_np)
    ctx = mp.get_context("spawn")
    # Single-threaded BLAS in every worker: the variables must be in the
    # environment the workers start with (numpy reads them on import).
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    os.environ.update({v: "1" for v in _THREAD_VARS})
    try:
        with ctx.Pool(cores, initializer=_init, initargs=(layout, kv_path, sm_scale, extra)) as pool:
            parts = pool.map(_shard, payloads, chunksize=1)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
        shutil.rmtree(tmp, ignore_errors=True)
    return {"tokens": sum(p["n"] for p in parts),
            "max_dout": max(p["max_dout"] for p in parts),
            "max_dlse": max(p["max_dlse"] for p in parts),
            "tight": max(p["tight"] for p in parts),
            "tight_full": max(p["tight_full"] for p in parts),
            "fail": next((p["fail"] for p in parts if p["fail"]), None)}


# ---------------------------------------------------------------------------
# the backward's heavily shared dkv rows, over every token that lists them
# ---------------------------------------------------------------------------

def _bits_to_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.array(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def _fwd_shard(payload):
    """Oracle forward of a shard: out as bf16 bits (rounded once, as the
    forward's output is) and the LSE as float32."""
    import torch
    from oracle import sparse_mla_oracle as orc
    toks, q_bits, idx = payload
    kv = _bits_to_bf16(np.asarray(_W["kv"]))
    o, l = orc.sparse_mla_fwd(_bits_to_bf16(q_bits), kv, torch.from_numpy(idx), _W["sm_scale"])
    return toks, _bits(torch.from_numpy(o).to(torch.bfloat16)), l.astype(np.float32)


def _bwd_rows_shard(payload):
    """The shard's tokens' contributions to dkv of the target rows, and of
    the per-element bounds of tests/parity.py (the backward given the oracle
    forward's out rounded to bf16)."""
    import torch
    from oracle import sparse_mla_oracle as orc
    from tests.parity import bf16_rounding_err, grad_term_bounds
    q_bits, idx, do_bits, rows = payload
    kv = _bits_to_bf16(np.asarray(_W["kv"]))
    q, dout, it = _bits_to_bf16(q_bits), _bits_to_bf16(do_bits), torch.from_numpy(idx)
    _, dkv = orc.sparse_mla_bwd(q, kv, it, _W["sm_scale"], dout)
    _, bkv = grad_term_bounds(q, kv, it, _W["sm_scale"], dout, bf16_rounding_err)
    return dkv[rows], bkv[rows]


def _dense_pool(kv, sm_scale, cores):
    import multiprocessing as mp
    tmp = tempfile.mkdtemp(prefix="oracle_pool_")
    path = os.path.join(tmp, "kv.npy")
    np.save(path, _bits(kv))
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    os.environ.update({v: "1" for v in _THREAD_VARS})
    try:
        pool = mp.get_context("spawn").Pool(cores or (os.cpu_count() or 1), initializer=_init,
                                            initargs=("dense", path, sm_scale, {}))
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    return pool, tmp


def oracle_fwd_dense_all(q, kv, indices, sm_scale: float, cores: int = 0, shard_tokens: int = 32):
    """The oracle forward of every token of a dense-layout workload on the
    host cores: (out bf16 [n, h, 512], lse float32 [n, h]) CPU tensors."""
    import torch
    n = q.shape[0]
    qb, idx = _bits(q), indices.reshape(n, -1).numpy().astype(np.int64)
    pool, tmp = _dense_pool(kv, sm_scale, cores)
    try:
        parts = pool.map(_fwd_shard, [(np.arange(a, min(n, a + shard_tokens)), qb[a:a + shard_tokens].copy(),
                                       idx[a:a + shard_tokens]) for a in range(0, n, shard_tokens)], chunksize=1)
    finally:
        pool.close()
        pool.join()
        shutil.rmtree(tmp, ignore_errors=True)
    out = np.concatenate([p[1] for p in parts])
    lse = np.concatenate([p[2] for p in parts])
    return _bits_to_bf16(out), torch.from_numpy(lse)


def oracle_bwd_dense_rows(q, kv, indices, dout, sm_scale: float, rows, cores: int = 0, shard_tokens: int = 32):
    """dkv of the given rows over every token of a dense-layout workload (the
    oracle's backward summed over token shards on the host cores), with the
    summed per-element bounds: (ref [R, 576], bound [R, 576]) float64."""
    n = q.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    qb, db = _bits(q), _bits(dout)
    idx = indices.reshape(n, -1).numpy().astype(np.int64)
    # only the tokens that list a target row contribute to it
    toks = np.nonzero(np.isin(idx, rows).any(axis=1))[0]
    pool, tmp = _dense_pool(kv, sm_scale, cores)
    try:
        parts = pool.map(_bwd_rows_shard, [(qb[toks[a:a + shard_tokens]], idx[toks[a:a + shard_tokens]],
                                            db[toks[a:a + shard_tokens]], rows)
                                           for a in range(0, toks.size, shard_tokens)], chunksize=1)
    finally:
        pool.close()
        pool.join()
        shutil.rmtree(tmp, ignore_errors=True)
    return sum(p[0] for p in parts), sum(p[1] for p in parts), int(toks.size)
