"""CPU float64 oracle for the DSA indexer and its top-k selection: the step
that produces the index lists the sparse-MLA forward consumes.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU baseline / reference arm use it.  It shares no code with
the CUDA path; both take their inputs from ``mla_inputs``.

Where it sits.  The pages name the indexer and its top-k as the producer of
the sparse lists ("[Feature] Add optional FlashMLA backend for DSA Sparse
MLA", Changes: the TileLang indexer is reused; "feat: add XTuner TileLang
sparse MLA backend", Summary: DSA index production is kept for short
prefill; Copilot overview: prefill scores are computed in query-row chunks
under a logits budget).  They do not print the score formula.  This module
reads it as the DSA "lightning indexer" published with DeepSeek-V3.2: per
query token t, indexer heads j < H_I with queries q[t,j,:] (D_I wide), one
indexer key k[s,:] per KV position s and per-token head weights w[t,j]

    I[t,s] = sum_j w[t,j] * max(0, q[t,j,:] . k[s,:])

over the positions t may see.  Causal visibility follows the forward's
indices-free mode: the s_q queries are the last s_q of s_kv positions, so
token t sees positions 0 .. t + s_kv - s_q, i.e.

    V(t) = clip(t + s_kv - s_q + 1, 0, s_kv)   positions.

Selection.  The index list of token t holds the topk visible positions of
largest I[t,s].  Three points the pages leave open, read here as:
  * equal scores are ranked by position, the smaller first (this makes the
    selected set unique);
  * the list is written in increasing position order and padded with -1 to
    topk entries (the forward is invariant to list order and reads -1 as
    masked);
  * a position whose score is -inf is not selectable: it is never listed,
    and a row with fewer than topk selectable positions lists those and pads
    with -1.  -inf is the mask of the attention's own score space (its
    fully masked row has LSE -inf), so such a position is one the attention
    could not use.
With V(t) <= topk every visible position is selected, so the list is
0 .. V(t)-1 then -1s, and no score is needed: the short-prefill rows of the
TileLang page's Summary.  Packed (varlen) prefill applies the same rules per
sequence with local positions, the convention of the packed forward; the
paged decode form reads a request's keys through its block table, with the
request's s_next MTP tokens at the end of its cache_seqlens positions (the
forward's decode convention).  A visible position whose page lies past the
block table's width, or whose table entry is outside [0, num_blocks), has no
key: it scores -inf and is never listed, short rows included.  The paged
forward masks exactly these positions (an index there reads no row), so the
indexer never lists an entry the forward would drop.

Pins (tests/test_indexer_oracle_pins.py): a worked example with small integers
whose scores and selection are computed by hand, positive homogeneity and
additivity in the weights, the ReLU's zero floor (a key anti-aligned with
every query scores exactly 0), selection against brute-force properties
(every selected score >= every unselected one, ties resolved to the smaller
positions), agreement with torch.topk on distinct scores, the short-row
identity lists, the packed form against the dense form per sequence, the
paged (decode) form against the packed form on a linearised cache and under a
shuffle of the physical pages, and the link to the forward: with every row
short, the sparse forward over these lists equals the indices-free causal
forward.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch


def _f64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def visible_len(t: int, s_q: int, s_kv: int) -> int:
    """Number of KV positions query t (0-based among the last s_q of s_kv
    positions) may see."""
    return int(min(max(t + s_kv - s_q + 1, 0), s_kv))


def token_scores(q_t: np.ndarray, w_t: np.ndarray, k_rows: np.ndarray) -> np.ndarray:
    """Indexer scores of one token over the given key rows.

    q_t [H_I, D_I], w_t [H_I], k_rows [n, D_I] (float64).  Returns [n]:
    sum over heads j of w_t[j] * relu(q_t[j] . k_rows[s])."""
    dots = q_t @ k_rows.T                    # [H_I, n]
    return (w_t[:, None] * np.maximum(dots, 0.0)).sum(axis=0)


def select_topk(scores: np.ndarray, topk: int) -> np.ndarray:
    """The topk positions of largest score, equal scores ranked by position
    (smaller first), listed in increasing position order and padded with -1.
    Positions scoring -inf are not selectable.  scores [V]; position p is
    scores[p]."""
    out = np.full(topk, -1, dtype=np.int64)
    cand = np.nonzero(~np.isneginf(scores))[0]
    if cand.size == 0:
        return out
    order = np.lexsort((cand, -scores[cand]))     # by score desc, then position asc
    take = np.sort(cand[order[:min(topk, cand.size)]])
    out[:take.shape[0]] = take
    return out


def identity_list(v: int, topk: int) -> np.ndarray:
    """The list of a short row (v <= topk visible positions): 0 .. v-1, then
    -1 to topk entries."""
    out = np.full(topk, -1, dtype=np.int64)
    out[:v] = np.arange(v)
    return out


def indexer_scores(q_idx, k_idx, weights, rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Dense causal prefill scores.  q_idx [s_q, H_I, D_I], k_idx [s_kv, D_I],
    weights [s_q, H_I].  Returns float64 [len(rows), s_kv] with -inf at the
    positions a token may not see (rows: the tokens, all by default)."""
    s_q, s_kv = q_idx.shape[0], k_idx.shape[0]
    k64 = _f64(k_idx)
    toks = range(s_q) if rows is None else list(rows)
    out = np.full((len(toks), s_kv), -np.inf)
    for i, t in enumerate(toks):
        v = visible_len(t, s_q, s_kv)
        if v:
            out[i, :v] = token_scores(_f64(q_idx[t]), _f64(weights[t]), k64[:v])
    return out


def dsa_indices(q_idx, k_idx, weights, topk: int, rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Dense causal prefill index lists [len(rows), topk] (int64, -1 padded):
    rows with V(t) <= topk get 0 .. V(t)-1, the others the top-k of their
    scores."""
    s_q, s_kv = q_idx.shape[0], k_idx.shape[0]
    k64 = _f64(k_idx)
    toks = range(s_q) if rows is None else list(rows)
    out = np.full((len(toks), topk), -1, dtype=np.int64)
    for i, t in enumerate(toks):
        v = visible_len(t, s_q, s_kv)
        if v <= topk:
            out[i] = identity_list(v, topk)
        else:
            out[i] = select_topk(token_scores(_f64(q_idx[t]), _f64(weights[t]), k64[:v]), topk)
    return out


def dsa_indices_varlen(q_idx, k_idx, weights, cu_seqlens_q, cu_seqlens_kv, topk: int,
                       rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Packed prefill: sequence b owns query rows cu_q[b] .. cu_q[b+1]-1 and
    KV rows cu_kv[b] .. cu_kv[b+1]-1; each token is scored and selected
    against its own sequence's keys with local positions (dense rules per
    sequence).  Returns int64 [len(rows), topk]."""
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_kv]
    total_q = cq[-1]
    toks = range(total_q) if rows is None else list(rows)
    out = np.full((len(toks), topk), -1, dtype=np.int64)
    for i, r in enumerate(toks):
        b = int(np.searchsorted(cq, r, side="right")) - 1
        lq, lk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
        t = r - cq[b]
        v = visible_len(t, lq, lk)
        if v <= topk:
            out[i] = identity_list(v, topk)
        else:
            ks = _f64(k_idx[ck[b]:ck[b] + v])
            out[i] = select_topk(token_scores(_f64(q_idx[r]), _f64(weights[r]), ks), topk)
    return out


def indexer_scores_varlen(q_idx, k_idx, weights, cu_seqlens_q, cu_seqlens_kv,
                          rows: Optional[Sequence[int]] = None, width: Optional[int] = None) -> np.ndarray:
    """Packed prefill scores: row i holds token rows[i]'s scores over its
    sequence's local positions 0 .. V-1, -inf beyond (width columns, default
    the longest KV sequence)."""
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_kv]
    if width is None:
        width = max(ck[b + 1] - ck[b] for b in range(len(ck) - 1))
    toks = range(cq[-1]) if rows is None else list(rows)
    out = np.full((len(toks), width), -np.inf)
    for i, r in enumerate(toks):
        b = int(np.searchsorted(cq, r, side="right")) - 1
        lq, lk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
        v = visible_len(r - cq[b], lq, lk)
        if v:
            out[i, :v] = token_scores(_f64(q_idx[r]), _f64(weights[r]), _f64(k_idx[ck[b]:ck[b] + v]))
    return out


def topk_rows(scores: np.ndarray, lens: Sequence[int], topk: int) -> np.ndarray:
    """Selection alone: row i's list from scores[i, :lens[i]] (lens[i] <= topk
    gives the identity list without reading scores).  Returns int64
    [rows, topk]."""
    out = np.full((scores.shape[0], topk), -1, dtype=np.int64)
    for i, v in enumerate(lens):
        v = int(v)
        if v <= topk:
            out[i] = identity_list(v, topk)
        else:
            out[i] = select_topk(np.asarray(scores[i, :v], dtype=np.float64), topk)
    return out


def page_valid(block_table, seqlen: int, page: int, num_blocks: int) -> np.ndarray:
    """bool [seqlen]: position s of the request has a key, i.e. its page
    s // page lies inside the block table and the table entry inside
    [0, num_blocks)."""
    bt = [int(x) for x in block_table]
    return np.array([s // page < len(bt) and 0 <= bt[s // page] < num_blocks for s in range(seqlen)],
                    dtype=bool)


def linearise_keys(k_cache, block_table, seqlen: int, page: int) -> np.ndarray:
    """The keys of one request in position order: position s is row s % page
    of physical block block_table[s // page] (a paged key cache laid out like
    the forward's paged KV cache).  Positions without a key (page_valid
    false) hold zeros here; their scores are -inf."""
    kc = _f64(k_cache)
    bt = [int(x) for x in block_table]
    zero = np.zeros(kc.shape[-1])

    def key(s):
        pg = s // page
        if pg >= len(bt) or not 0 <= bt[pg] < kc.shape[0]:
            return zero
        return kc[bt[pg], s % page]
    rows = [key(s) for s in range(seqlen)]
    return np.stack(rows) if rows else np.zeros((0, kc.shape[-1]))


def paged_row_scores(q_t, w_t, keys: np.ndarray, valid: np.ndarray) -> np.ndarray:
    """Scores of one decode row over its visible positions (keys [v, D_I],
    valid [v]): the indexer score where the position has a key, -inf
    elsewhere."""
    sc = token_scores(q_t, w_t, keys)
    sc[~valid] = -np.inf
    return sc


def dsa_indices_paged(q_idx, k_cache, weights, block_table, cache_seqlens, topk: int, page: int,
                      rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Decode: request b has s_next query rows b s_next .. b s_next + s_next - 1
    at the end of its cache_seqlens[b] positions (MTP token j sits at
    position L_b - s_next + j and sees positions 0 .. L_b - s_next + j), its
    keys in the paged cache k_cache [num_blocks, page, D_I] through
    block_table [batch, max_blocks].  The dense rules per request on its
    linearised keys.  q_idx [batch, s_next, H_I, D_I], weights
    [batch, s_next, H_I].  Returns int64 [len(rows), topk] over the flattened
    rows b s_next + j."""
    batch, s_next = q_idx.shape[0], q_idx.shape[1]
    q2 = q_idx.reshape(batch * s_next, *q_idx.shape[2:])
    w2 = weights.reshape(batch * s_next, -1)
    toks = range(batch * s_next) if rows is None else list(rows)
    out = np.full((len(toks), topk), -1, dtype=np.int64)
    keys = {}
    num_blocks = k_cache.shape[0]
    for i, r in enumerate(toks):
        b, j = divmod(r, s_next)
        lk = int(cache_seqlens[b])
        v = visible_len(j, s_next, lk)
        ok = page_valid(block_table[b], v, page, num_blocks)
        if v <= topk:   # every position with a key, in order
            pos = np.nonzero(ok)[0]
            out[i, :pos.size] = pos
            continue
        if b not in keys:
            keys[b] = linearise_keys(k_cache, block_table[b], lk, page)
        out[i] = select_topk(paged_row_scores(_f64(q2[r]), _f64(w2[r]), keys[b][:v], ok), topk)
    return out
