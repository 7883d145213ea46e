"""CPU float64 oracle for the DSA sparse-MLA attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU baseline / reference arm use it.  It shares no code with
the CUDA path; both take their inputs from ``mla_inputs``.

What it computes (plain definition, float64, from the exact bf16 inputs):

For query token t, head h and index list I_t of length topk, the valid
entries are those that are not -1 and lie inside the token's KV range
("feat: add XTuner TileLang sparse MLA backend", Validation: outputs include
-1-padded index lists; out-of-range entries are read as masked as well).
Each valid entry j maps to a KV row r_j of the single shared latent head
("[Feature] Add optional FlashMLA backend for DSA Sparse MLA", Runtime
constraints: kv_group=1, value_dim=512).  With d_qk=576 and d_v=512 (the
TileLang page, Performance, Isolated sparse MLA forward):

    s_{h,j}   = sm_scale * sum_{d<576} q[t,h,d] * kv[r_j,d]
    LSE[t,h]  = log sum_{j valid} exp(s_{h,j})               (natural log)
    out[t,h,:] = sum_{j valid} exp(s_{h,j} - LSE[t,h]) * kv[r_j, 0:512]

A list with no valid entry gives out = 0 and LSE = -inf.  Entries are taken
with multiplicity (a repeated index counts once per occurrence).  The value
is the first 512 columns of the same latent row.  Output and LSE are the two
results the FlashMLA page aligns between implementations (Motivation).

Row mapping per entry point ("feat: add XTuner TileLang sparse MLA backend",
Summary: packed prefill and zero-copy BF16 paged-cache decode share one
kernel; Copilot overview: sparse index mapping to cache slots):

* dense prefill:  r = idx, valid iff 0 <= idx < s_kv;
* packed prefill: r = cu_seqlens_kv[b] + idx, valid iff
  0 <= idx < cu_seqlens_kv[b+1] - cu_seqlens_kv[b], b the token's sequence;
* paged decode:   r = block_table[b, idx // page] * page + idx % page,
  valid iff 0 <= idx < cache_seqlens[b] and the page entry lies in the pool.

Pins (tests/test_oracle_pins.py): a dense multiplicity-matrix formulation
with torch.logsumexp on tiny inputs, dense causal attention through
torch's scaled_dot_product_attention when every causal position is listed,
invariance to index order and to -1 padding, closed forms (single valid
entry, zero query, duplicated entry, all masked) and the logsumexp
definition.  Packed and paged variants are pinned against dense causal
attention per sequence and against the dense-layout oracle on a linearised
cache.  The indices-free causal mode is pinned against torch's
scaled_dot_product_attention (causal, and with an explicit bottom-right mask
when the queries are the last s_q of s_kv positions).  The backward is pinned
against torch autograd through an independent dense formulation of the
forward, and against central finite differences on a tiny case.
"""
from __future__ import annotations

from typing import Iterable, Optional, Sequence, Tuple

import numpy as np
import torch

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Exact upcast of a bf16/float tensor (or array) to float64."""
    if isinstance(x, torch.Tensor):
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


def attend(q_t: np.ndarray, rows: np.ndarray, sm_scale: float, d_v: int
           ) -> Tuple[np.ndarray, np.ndarray]:
    """Scaled softmax attention of one token's heads over its gathered rows.

    q_t [h, d_qk] float64; rows [n, d_qk] float64 (the valid entries, in list
    order, with multiplicity).  Returns out [h, d_v] and lse [h].
    """
    h = q_t.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((h, d_v)), np.full(h, NEG_INF)
    s = sm_scale * (q_t @ rows.T)                      # [h, n]
    m = s.max(axis=1, keepdims=True)
    lse = m + np.log(np.exp(s - m).sum(axis=1, keepdims=True))
    p = np.exp(s - lse)                                # softmax weights
    out = p @ rows[:, :d_v]
    return out, lse[:, 0]


# --------------------------------------------------------------------------
# row selection (valid entries -> KV rows)
# --------------------------------------------------------------------------

def rows_dense(idx_t: np.ndarray, s_kv: int) -> np.ndarray:
    v = idx_t[(idx_t != -1) & (idx_t >= 0) & (idx_t < s_kv)]
    return v


def rows_varlen(idx_t: np.ndarray, kv_start: int, kv_len: int) -> np.ndarray:
    v = idx_t[(idx_t != -1) & (idx_t >= 0) & (idx_t < kv_len)]
    return kv_start + v


def rows_paged(idx_t: np.ndarray, table_b: np.ndarray, seqlen: int, page: int,
               num_blocks: int) -> np.ndarray:
    v = idx_t[(idx_t != -1) & (idx_t >= 0) & (idx_t < seqlen)]
    pg = v // page
    ok = pg < table_b.shape[0]
    v, pg = v[ok], pg[ok]
    blk = table_b[pg]
    ok = (blk >= 0) & (blk < num_blocks)
    return blk[ok] * page + (v[ok] % page)


def _gather(kv, rows: np.ndarray) -> np.ndarray:
    if isinstance(kv, torch.Tensor):
        return _f64(kv[torch.from_numpy(rows)])
    return kv[rows]


# --------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------

def sparse_mla_fwd(q, kv, indices, sm_scale: float, d_v: int = 512,
                   tokens: Optional[Iterable[int]] = None):
    """Dense-layout forward.  q [s_q,h,576], kv [s_kv,576] (or [s_kv,1,576]),
    indices [s_q,topk] (or [s_q,1,topk]).  Returns float64 (out, lse) for the
    requested tokens (all by default), stacked in request order."""
    s_q = q.shape[0]
    kv2 = kv.reshape(kv.shape[0], -1)
    idx = _i64(indices).reshape(s_q, -1)
    toks = range(s_q) if tokens is None else list(tokens)
    outs, lses = [], []
    for t in toks:
        r = rows_dense(idx[t], kv2.shape[0])
        o, l = attend(_f64(q[t]), _gather(kv2, r), sm_scale, d_v)
        outs.append(o)
        lses.append(l)
    return _stack(outs, lses, q.shape[1], d_v)


def sequence_of(cu_seqlens_q, t: int) -> int:
    """Index b with cu_q[b] <= t < cu_q[b+1]."""
    cu = _i64(cu_seqlens_q)
    return int(np.searchsorted(cu, t, side="right") - 1)


def sparse_mla_fwd_varlen(q, kv, indices, cu_seqlens_q, cu_seqlens_kv, sm_scale: float,
                          d_v: int = 512, tokens: Optional[Iterable[int]] = None):
    """Packed prefill; indices are local to each token's own sequence."""
    total = q.shape[0]
    kv2 = kv.reshape(kv.shape[0], -1)
    idx = _i64(indices).reshape(total, -1)
    cu_q = _i64(cu_seqlens_q)
    cu_k = _i64(cu_seqlens_kv)
    toks = range(total) if tokens is None else list(tokens)
    outs, lses = [], []
    for t in toks:
        b = int(np.searchsorted(cu_q, t, side="right") - 1)
        r = rows_varlen(idx[t], int(cu_k[b]), int(cu_k[b + 1] - cu_k[b]))
        o, l = attend(_f64(q[t]), _gather(kv2, r), sm_scale, d_v)
        outs.append(o)
        lses.append(l)
    return _stack(outs, lses, q.shape[1], d_v)


def sparse_mla_decode(q, kv_cache, block_table, cache_seqlens, indices, sm_scale: float,
                      page_size: int = 64, d_v: int = 512,
                      tokens: Optional[Iterable[Tuple[int, int]]] = None):
    """Paged decode.  q [b,s_next,h,576]; kv_cache [num_blocks,page,576];
    indices [b,s_next,topk] logical positions.  ``tokens`` is a list of
    (request, slot) pairs; results come back as [n, h, d_v] / [n, h]."""
    batch, s_next, h = q.shape[0], q.shape[1], q.shape[2]
    num_blocks = kv_cache.shape[0]
    flat = kv_cache.reshape(num_blocks * page_size, -1)
    table = _i64(block_table)
    lens = _i64(cache_seqlens)
    idx = _i64(indices).reshape(batch, s_next, -1)
    toks = [(b, j) for b in range(batch) for j in range(s_next)] if tokens is None else list(tokens)
    outs, lses = [], []
    for b, j in toks:
        r = rows_paged(idx[b, j], table[b], int(lens[b]), page_size, num_blocks)
        o, l = attend(_f64(q[b, j]), _gather(flat, r), sm_scale, d_v)
        outs.append(o)
        lses.append(l)
    return _stack(outs, lses, h, d_v)


def causal_mla_fwd(q, kv, sm_scale: float, d_v: int = 512,
                   tokens: Optional[Iterable[int]] = None):
    """Indices-free causal forward, the short-prefill case where every causal
    position is selected ("feat: add XTuner TileLang sparse MLA backend",
    Summary: short prefill keeps DSA index production; with s <= topk the
    top-k list of token t is all of positions 0..t).  q [s_q,h,576], kv
    [s_kv,576].  Query t sits at position t + s_kv - s_q (the queries are the
    last s_q positions) and attends to every KV row at or before it; a query
    before position 0 attends to nothing.  Returns float64 (out, lse)."""
    s_q = q.shape[0]
    kv2 = kv.reshape(kv.shape[0], -1)
    s_kv = kv2.shape[0]
    toks = range(s_q) if tokens is None else list(tokens)
    outs, lses = [], []
    for t in toks:
        last = t + s_kv - s_q
        r = np.arange(0, max(0, min(last + 1, s_kv)), dtype=np.int64)
        o, l = attend(_f64(q[t]), _gather(kv2, r), sm_scale, d_v)
        outs.append(o)
        lses.append(l)
    return _stack(outs, lses, q.shape[1], d_v)


def bwd_token(q_t: np.ndarray, K: np.ndarray, do_t: np.ndarray, sm_scale: float, d_v: int
              ) -> Tuple[np.ndarray, np.ndarray]:
    """One token's backward over its gathered rows K [n, 576] (V = K[:, :512],
    the same latent rows), from the definition of the forward by the chain
    rule (the LSE output carries no gradient):

        P  = softmax(sm_scale * q_t K^T)            [h, n]
        dP = dout_t V^T                             [h, n]
        D  = rowsum(dout_t * out_t) = rowsum(P * dP)
        dS = P * (dP - D)
        dq_t  = sm_scale * dS K                     [h, 576]
        dK    = sm_scale * dS^T q_t, plus P^T dout_t on the first 512 columns

    Returns (dq_t, dK [n, 576]); the caller adds dK into the rows."""
    V = K[:, :d_v]
    s = sm_scale * (q_t @ K.T)
    m = s.max(axis=1, keepdims=True)
    P = np.exp(s - m)
    P /= P.sum(axis=1, keepdims=True)
    O = P @ V
    dP = do_t @ V.T
    D = (do_t * O).sum(axis=1, keepdims=True)
    dS = P * (dP - D)
    dK = sm_scale * (dS.T @ q_t)
    dK[:, :d_v] += P.T @ do_t
    return sm_scale * (dS @ K), dK


def sparse_mla_bwd(q, kv, indices, sm_scale: float, dout, d_v: int = 512):
    """Gradients of the dense-layout forward with respect to q and kv, given
    the upstream gradient dout of out: the backward the training users pair
    with the forward (prime-rl page: forward and backward sparse attention
    timings).  Per token, bwd_token over its valid rows, with multiplicity (a
    row listed twice receives both contributions).  O and the LSE are
    recomputed from q and kv.  Returns float64 dq [s_q,h,576], dkv [s_kv,576]."""
    s_q, h = q.shape[0], q.shape[1]
    kv2 = kv.reshape(kv.shape[0], -1)
    s_kv, d_qk = kv2.shape
    idx = _i64(indices).reshape(s_q, -1)
    q64, do64 = _f64(q), _f64(dout)
    dq = np.zeros((s_q, h, d_qk))
    dkv = np.zeros((s_kv, d_qk))
    for t in range(s_q):
        r = rows_dense(idx[t], s_kv)
        if r.size == 0:
            continue
        dq[t], dK = bwd_token(q64[t], _gather(kv2, r), do64[t], sm_scale, d_v)
        np.add.at(dkv, r, dK)
    return dq, dkv


def sparse_mla_bwd_varlen(q, kv, indices, cu_seqlens_q, cu_seqlens_kv, sm_scale: float, dout,
                          d_v: int = 512):
    """Packed-prefill backward: as sparse_mla_bwd with each token's local
    indices mapped into its own sequence's KV rows (rows_varlen)."""
    total = q.shape[0]
    h = q.shape[1]
    kv2 = kv.reshape(kv.shape[0], -1)
    n_rows, d_qk = kv2.shape
    idx = _i64(indices).reshape(total, -1)
    cu_q, cu_k = _i64(cu_seqlens_q), _i64(cu_seqlens_kv)
    q64, do64 = _f64(q), _f64(dout)
    dq = np.zeros((total, h, d_qk))
    dkv = np.zeros((n_rows, d_qk))
    for t in range(total):
        b = sequence_of(cu_q, t)
        r = rows_varlen(idx[t], int(cu_k[b]), int(cu_k[b + 1] - cu_k[b]))
        if r.size == 0:
            continue
        dq[t], dK = bwd_token(q64[t], _gather(kv2, r), do64[t], sm_scale, d_v)
        np.add.at(dkv, r, dK)
    return dq, dkv


def valid_count_dense(indices, s_kv: int) -> np.ndarray:
    """|V_t| per token: the number of valid entries, with multiplicity."""
    idx = _i64(indices).reshape(indices.shape[0], -1)
    return np.array([rows_dense(r, s_kv).size for r in idx], dtype=np.int64)


def valid_count_varlen(indices, cu_seqlens_q, cu_seqlens_kv) -> np.ndarray:
    """|V_t| per packed token (entries local to the token's sequence)."""
    idx = _i64(indices).reshape(indices.shape[0], -1)
    cu_q, cu_k = _i64(cu_seqlens_q), _i64(cu_seqlens_kv)
    out = np.zeros(idx.shape[0], dtype=np.int64)
    for t in range(idx.shape[0]):
        b = int(np.searchsorted(cu_q, t, side="right") - 1)
        out[t] = rows_varlen(idx[t], int(cu_k[b]), int(cu_k[b + 1] - cu_k[b])).size
    return out


def valid_count_paged(indices, block_table, cache_seqlens, page_size: int, num_blocks: int) -> np.ndarray:
    """|V_t| per decode token, flattened as [batch * s_next]."""
    table = _i64(block_table)
    lens = _i64(cache_seqlens)
    batch = table.shape[0]
    idx = _i64(indices).reshape(batch, -1, indices.shape[-1])
    return np.array([rows_paged(idx[b, j], table[b], int(lens[b]), page_size, num_blocks).size
                     for b in range(batch) for j in range(idx.shape[1])], dtype=np.int64)


def _stack(outs, lses, h, d_v):
    if not outs:
        return np.zeros((0, h, d_v)), np.zeros((0, h))
    return np.stack(outs), np.stack(lses)
