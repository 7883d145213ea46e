"""Seeded synthetic inputs for the DSA sparse-MLA forward.

This module builds inputs only: Q, the latent KV rows, the top-k index
lists, packing offsets and the paged cache with its block table.  It holds
none of the attention arithmetic; the oracle and the CUDA path both consume
what it returns and neither is imported here.

Shapes and index structure follow the workloads of the pages:

* one shared latent KV head of 576 bf16 values per token whose first 512
  are the value ("[Feature] Add optional FlashMLA backend for DSA Sparse
  MLA", Runtime constraints: kv_group=1, value_dim=512);
* dqk=576, dv=512, topk=2048 at 8 TP-local query heads
  ("feat: add XTuner TileLang sparse MLA backend", Performance, Isolated
  sparse MLA forward), with -1 padded index lists (same page, Validation);
* packed prefill and a BF16 paged cache for decode (same page, Summary);
* MTP5 speculative decode, six query tokens per request (same page,
  End-to-end serving);
* the DSA indexer that produces the lists (the pages name it but print
  neither its formula nor its sizes): 64 indexer heads of width 128, one
  key per position and per-token head weights, the sizes of the DeepSeek-V3.2
  lightning indexer.

Recipe: Q and KV are float32 standard normal draws from a CPU
``torch.Generator`` seeded per case, rounded to bf16 (round to nearest
even).  Index lists draw distinct causal positions with ``torch.randperm``
from generators derived from the same seed.  Indexer queries and keys are
N(0,1) draws rounded to bf16; head weights are fp32 N(0,1) draws scaled by
h_idx^-1/2 * d_idx^-1/2.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

D_QK = 576
D_V = 512
TOPK = 2048
PAGE = 64


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(g: torch.Generator, shape) -> torch.Tensor:
    """float32 N(0,1) draws rounded to bf16 (RNE)."""
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def default_sm_scale(d_qk: int = D_QK) -> float:
    """1/sqrt(d_qk): the scale the workloads use (576 -> 1/24)."""
    return 1.0 / math.sqrt(d_qk)


# --------------------------------------------------------------------------
# index-list patterns (each returns the picked positions of one query row)
# --------------------------------------------------------------------------

def pick_causal(g: torch.Generator, i: int, topk: int) -> torch.Tensor:
    """min(i+1, topk) distinct positions drawn uniformly from [0, i]."""
    return torch.randperm(i + 1, generator=g)[: min(i + 1, topk)].to(torch.int32)


def pick_recent(g: torch.Generator, i: int, topk: int, recent: int = 128) -> torch.Tensor:
    """The min(recent, i+1) most recent positions i, i-1, ... first, then
    min(i+1, topk) - recent distinct uniform positions from [0, i-recent]."""
    n_recent = min(recent, i + 1)
    head = torch.arange(i, i - n_recent, -1, dtype=torch.int32)
    n_rest = min(i + 1, topk) - n_recent
    if n_rest <= 0:
        return head
    tail = torch.randperm(i + 1 - recent, generator=g)[:n_rest].to(torch.int32)
    return torch.cat([head, tail])


def pad_rows(rows: List[torch.Tensor], topk: int) -> torch.Tensor:
    out = torch.full((len(rows), topk), -1, dtype=torch.int32)
    for t, r in enumerate(rows):
        out[t, : r.numel()] = r
    return out


# --------------------------------------------------------------------------
# cases
# --------------------------------------------------------------------------

@dataclass
class PrefillCase:
    """Inputs of one dense-layout forward call.

    q [s_q, h_q, d_qk] bf16, kv [s_kv, d_qk] bf16 (the single latent head),
    indices [s_q, topk] int32 (-1 padded).  ``referenced`` lists the KV rows
    the generator placed in some index list (used to poison every other row).
    """
    name: str
    q: torch.Tensor
    kv: torch.Tensor
    indices: torch.Tensor
    sm_scale: float
    d_v: int = D_V
    referenced: Optional[torch.Tensor] = None

    @property
    def s_q(self):
        return self.q.shape[0]

    @property
    def h_q(self):
        return self.q.shape[1]

    @property
    def s_kv(self):
        return self.kv.shape[0]

    @property
    def topk(self):
        return self.indices.shape[1]


@dataclass
class VarlenCase:
    """Packed prefill: sequences concatenated along the token axis.

    cu_seqlens_q / cu_seqlens_kv [batch+1] int32; indices are local to the
    query token's own sequence.
    """
    name: str
    q: torch.Tensor
    kv: torch.Tensor
    indices: torch.Tensor
    cu_seqlens_q: torch.Tensor
    cu_seqlens_kv: torch.Tensor
    sm_scale: float
    d_v: int = D_V
    referenced: Optional[torch.Tensor] = None

    @property
    def batch(self):
        return self.cu_seqlens_q.numel() - 1


@dataclass
class DecodeCase:
    """Paged-cache decode.

    q [batch, s_next, h_q, d_qk]; kv_cache [num_blocks, page, d_qk];
    block_table [batch, max_blocks] int32; cache_seqlens [batch] int32;
    indices [batch, s_next, topk] int32 logical positions in the request.
    """
    name: str
    q: torch.Tensor
    kv_cache: torch.Tensor
    block_table: torch.Tensor
    cache_seqlens: torch.Tensor
    indices: torch.Tensor
    sm_scale: float
    page_size: int = PAGE
    d_v: int = D_V
    picked: List[torch.Tensor] = field(default_factory=list)

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def s_next(self):
        return self.q.shape[1]

    @property
    def h_q(self):
        return self.q.shape[2]


def prefill_indices(seed: int, s_q: int, s_kv: int, topk: int = TOPK,
                    pattern: str = "causal") -> torch.Tensor:
    """[s_q, topk] int32 causal index lists (query i picks from [0, i])."""
    gi = _gen(seed * 7919 + 17)
    rows = []
    for i in range(s_q):
        last = min(i, s_kv - 1)
        if pattern == "causal":
            rows.append(pick_causal(gi, last, topk))
        elif pattern == "recent":
            rows.append(pick_recent(gi, last, topk))
        else:
            raise ValueError(pattern)
    return pad_rows(rows, topk)


def prefill_case(seed: int, s_q: int, s_kv: int, h_q: int, topk: int = TOPK,
                 pattern: str = "causal", d_qk: int = D_QK, d_v: int = D_V,
                 name: str = "") -> PrefillCase:
    """Causal prefill: query i picks positions from [0, i] (i < s_kv)."""
    g = _gen(seed)
    q = randn_bf16(g, (s_q, h_q, d_qk))
    kv = randn_bf16(g, (s_kv, d_qk))
    idx = prefill_indices(seed, s_q, s_kv, topk, pattern)
    ref = torch.unique(idx[idx >= 0])
    return PrefillCase(name or f"prefill_s{s_q}_h{h_q}", q, kv, idx,
                       default_sm_scale(d_qk), d_v, ref)


def varlen_indices(seed: int, seqlens: List[int], topk: int = TOPK):
    """Local causal index lists for packed sequences; returns
    (indices [total, topk] int32, cu_seqlens [batch+1] int32,
    referenced global rows)."""
    gi = _gen(seed * 7919 + 17)
    rows, refs = [], []
    cu = [0]
    for L in seqlens:
        for i in range(L):
            r = pick_causal(gi, i, topk)
            rows.append(r)
            refs.append(r.to(torch.int64) + cu[-1])
        cu.append(cu[-1] + L)
    idx = pad_rows(rows, topk)
    cu_t = torch.tensor(cu, dtype=torch.int32)
    ref = torch.unique(torch.cat(refs)) if refs else torch.empty(0, dtype=torch.int64)
    return idx, cu_t, ref


def varlen_case(seed: int, seqlens: List[int], h_q: int, topk: int = TOPK,
                d_qk: int = D_QK, name: str = "") -> VarlenCase:
    """Packed prefill; each sequence causal within itself (local indices)."""
    g = _gen(seed)
    total = int(sum(seqlens))
    q = randn_bf16(g, (total, h_q, d_qk))
    kv = randn_bf16(g, (total, d_qk))
    idx, cu_t, ref = varlen_indices(seed, seqlens, topk)
    return VarlenCase(name or f"varlen_{total}_h{h_q}", q, kv, idx, cu_t, cu_t.clone(),
                      default_sm_scale(d_qk), D_V, ref)


def decode_case(seed: int, batch: int, s_next: int, h_q: int, lo: int, hi: int,
                topk: int = TOPK, page: int = PAGE, spare_pages: int = 64,
                d_qk: int = D_QK, poison: bool = True, name: str = "") -> DecodeCase:
    """Paged decode with MTP-style speculative tokens.

    Request b has context length L_b ~ U[lo, hi]; its s_next query tokens sit
    at positions L_b - s_next ... L_b - 1 and token j picks topk distinct
    positions uniformly from [0, L_b - s_next + j].  The page pool holds
    sum(ceil(L_b / page)) + spare_pages pages in a random order (the block
    table is a random permutation).  With ``poison`` every cache slot that no
    index list picks is set to NaN, so any read of it shows up in the result.
    """
    g = _gen(seed)
    lens = torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64)
    n_pages = [int(math.ceil(int(L) / page)) for L in lens]
    num_blocks = sum(n_pages) + spare_pages
    max_blocks = max(n_pages)
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    block_table = torch.zeros((batch, max_blocks), dtype=torch.int32)
    off = 0
    for b in range(batch):
        block_table[b, : n_pages[b]] = perm[off: off + n_pages[b]]
        off += n_pages[b]
    q = randn_bf16(g, (batch, s_next, h_q, d_qk))
    kv_cache = randn_bf16(g, (num_blocks, page, d_qk))
    gi = _gen(seed * 7919 + 17)
    idx = torch.full((batch, s_next, topk), -1, dtype=torch.int32)
    picked = []
    for b in range(batch):
        L = int(lens[b])
        for j in range(s_next):
            last = L - s_next + j
            r = pick_causal(gi, last, topk)
            idx[b, j, : r.numel()] = r
            picked.append(r)
    if poison:
        keep = torch.zeros(num_blocks * page, dtype=torch.bool)
        for b in range(batch):
            pos = torch.unique(idx[b][idx[b] >= 0]).to(torch.int64)
            slots = block_table[b, pos // page].to(torch.int64) * page + pos % page
            keep[slots] = True
        flat = kv_cache.view(-1, d_qk)
        flat[~keep] = float("nan")
    return DecodeCase(name or f"decode_b{batch}_s{s_next}_h{h_q}", q, kv_cache, block_table,
                      lens.to(torch.int32), idx, default_sm_scale(d_qk), page, D_V, picked)


def poison_unreferenced(kv: torch.Tensor, referenced: torch.Tensor) -> torch.Tensor:
    """Copy of ``kv`` with every row not in ``referenced`` set to NaN."""
    out = kv.clone()
    mask = torch.ones(kv.shape[0], dtype=torch.bool)
    if referenced is not None and referenced.numel():
        mask[referenced.to(torch.int64)] = False
    out[mask] = float("nan")
    return out


def scatter_padding(g: torch.Generator, indices: torch.Tensor) -> torch.Tensor:
    """Shuffle each row so -1 entries sit anywhere, not only at the end."""
    out = indices.clone()
    flat = out.view(-1, out.shape[-1])
    for t in range(flat.shape[0]):
        flat[t] = flat[t, torch.randperm(flat.shape[1], generator=g)]
    return out


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

VARLEN_C4 = [8192, 4096, 2048, 1024, 1024]


def config(n: int, seed: Optional[int] = None):
    """Workload n (1..5) with seed 1000+n unless given."""
    seed = 1000 + n if seed is None else seed
    if n == 1:
        return prefill_case(seed, 64, 64, 8, name="c1_tiny_prefill_s64_h8")
    if n == 2:
        return prefill_case(seed, 2119, 2119, 8, name="c2_mid_prefill_s2119_h8")
    if n == 3:
        return prefill_case(seed, 8192, 8192, 64, pattern="recent",
                            name="c3_wide_prefill_s8192_h64")
    if n == 4:
        return varlen_case(seed, VARLEN_C4, 64, name="c4_varlen_16384_h64")
    if n == 5:
        return decode_case(seed, 16, 6, 8, 4096, 32768, name="c5_paged_decode_b16_mtp6_h8")
    raise ValueError(n)


# --------------------------------------------------------------------------
# FP8 KV cache (the cache writer's quantization; the decode reads it)
# --------------------------------------------------------------------------

FP8_SLOT_BYTES = 656   # 512 e4m3 codes, 4 fp32 tile scales, 64 bf16 rope values


def quantize_fp8_slots(latent: torch.Tensor, pow2_scales: bool = False) -> torch.Tensor:
    """Latent rows [..., 576] -> FP8 cache slots uint8 [..., 656] in the
    layout of DeepSeek-V3.2's FP8 sparse-decode cache: the first 512 values
    as float8 e4m3 codes in four tiles of 128, each with an fp32 scale
    amax / 448 (rounded up to a power of two with ``pow2_scales``), then the
    scales, then the last 64 values as bf16.  The codes come from torch's
    float8_e4m3fn conversion (round to nearest even).  A row holding NaN
    (a poisoned slot) gets NaN codes, scales and rope values."""
    lead = latent.shape[:-1]
    x = latent.float().reshape(-1, D_QK)
    v = x[:, :512].reshape(-1, 4, 128)
    amax = v.abs().amax(dim=-1)
    scale = amax / 448.0
    scale = torch.where(scale > 0, scale, torch.ones_like(scale))
    if pow2_scales:
        scale = torch.exp2(torch.ceil(torch.log2(scale)))
    scale = torch.where(torch.isnan(amax), torch.full_like(scale, float("nan")), scale)
    codes = (v / scale[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(-1, 512)
    sc = scale.to(torch.float32).contiguous().view(torch.uint8).reshape(-1, 16)
    rope = x[:, 512:].to(torch.bfloat16).contiguous().view(torch.uint8).reshape(-1, 128)
    return torch.cat([codes, sc, rope], dim=1).reshape(*lead, FP8_SLOT_BYTES).contiguous()


def decode_case_fp8(seed: int, batch: int, s_next: int, h_q: int, lo: int, hi: int, topk: int = TOPK,
                    page: int = PAGE, spare_pages: int = 64, pow2_scales: bool = False, name: str = ""):
    """A paged decode case whose cache is FP8: decode_case's structure
    (contexts, shuffled pool, index lists, NaN in every slot no list picks),
    its latent rows written as FP8 slots.  Returns (case, cache_u8 [num_blocks,
    page, 656])."""
    c = decode_case(seed, batch, s_next, h_q, lo, hi, topk=topk, page=page, spare_pages=spare_pages,
                    name=name or f"decode_fp8_b{batch}_s{s_next}_h{h_q}")
    return c, quantize_fp8_slots(c.kv_cache, pow2_scales=pow2_scales)


def nominal_flops(s_q: int, h_q: int, topk: int = TOPK, d_qk: int = D_QK, d_v: int = D_V) -> float:
    """2*s_q*h_q*topk*(d_qk+d_v): the workload's nominal FLOP count."""
    return 2.0 * s_q * h_q * topk * (d_qk + d_v)


# --------------------------------------------------------------------------
# DSA indexer inputs (the step that produces the index lists)
# --------------------------------------------------------------------------

H_IDX = 64     # indexer heads
D_IDX = 128    # indexer head width


@dataclass
class IndexerCase:
    """Indexer queries q_idx [total_q, h_idx, d_idx] bf16, one key per KV
    position k_idx [total_kv, d_idx] bf16 and per-token head weights
    [total_q, h_idx] fp32.  cu_seqlens_q / cu_seqlens_kv (int32 [batch+1])
    are None for a dense prefill (one sequence)."""
    name: str
    q_idx: torch.Tensor
    k_idx: torch.Tensor
    weights: torch.Tensor
    topk: int
    cu_seqlens_q: Optional[torch.Tensor] = None
    cu_seqlens_kv: Optional[torch.Tensor] = None

    @property
    def max_seqlen_kv(self) -> int:
        if self.cu_seqlens_kv is None:
            return int(self.k_idx.shape[0])
        return int((self.cu_seqlens_kv[1:] - self.cu_seqlens_kv[:-1]).max().item())


def indexer_weights(g: torch.Generator, total_q: int, h_idx: int, d_idx: int) -> torch.Tensor:
    """Head weights: N(0,1) draws times h_idx^-1/2 * d_idx^-1/2 (a projection
    of the hidden state folded with the head-count and softmax scales), fp32."""
    w = torch.randn((total_q, h_idx), generator=g, dtype=torch.float32)
    return w * float(h_idx ** -0.5 * d_idx ** -0.5)


def indexer_case(seed: int, s_q: int, s_kv: int, h_idx: int = H_IDX, d_idx: int = D_IDX,
                 topk: int = TOPK, name: str = "") -> IndexerCase:
    """Dense causal prefill: the s_q queries are the last s_q of s_kv
    positions.  q_idx, k_idx N(0,1) rounded to bf16."""
    g = _gen(seed * 104729 + 3)
    q = randn_bf16(g, (s_q, h_idx, d_idx))
    k = randn_bf16(g, (s_kv, d_idx))
    w = indexer_weights(g, s_q, h_idx, d_idx)
    return IndexerCase(name or f"indexer_s{s_q}_kv{s_kv}_h{h_idx}", q, k, w, topk)


def indexer_varlen_case(seed: int, q_lens: List[int], kv_lens: List[int], h_idx: int = H_IDX,
                        d_idx: int = D_IDX, topk: int = TOPK, name: str = "") -> IndexerCase:
    """Packed prefill: sequence b has q_lens[b] new tokens at the end of
    kv_lens[b] positions (kv_lens[b] - q_lens[b] cached before them)."""
    assert len(q_lens) == len(kv_lens)
    g = _gen(seed * 104729 + 5)
    tq, tk = int(sum(q_lens)), int(sum(kv_lens))
    q = randn_bf16(g, (tq, h_idx, d_idx))
    k = randn_bf16(g, (tk, d_idx))
    w = indexer_weights(g, tq, h_idx, d_idx)
    cq = torch.tensor([0] + list(torch.cumsum(torch.tensor(q_lens), 0).tolist()), dtype=torch.int32)
    ck = torch.tensor([0] + list(torch.cumsum(torch.tensor(kv_lens), 0).tolist()), dtype=torch.int32)
    return IndexerCase(name or f"indexer_varlen_{tq}_{tk}_h{h_idx}", q, k, w, topk, cq, ck)


def tied_scores(seed: int, rows: int, width: int, levels: int = 7) -> torch.Tensor:
    """Scores fp32 [rows, width] drawn from a few integer levels (many exact
    ties) with some -inf entries, for the selection step alone."""
    g = _gen(seed * 7 + 11)
    s = torch.randint(-levels, levels + 1, (rows, width), generator=g).to(torch.float32)
    hole = torch.rand((rows, width), generator=g) < 0.02
    s[hole] = float("-inf")
    return s


@dataclass
class IndexerPagedCase:
    """Decode indexer inputs: q_idx [batch, s_next, h_idx, d_idx] bf16, a
    paged key cache k_cache [num_blocks, page, d_idx] bf16 with its
    block_table [batch, max_blocks] int32 and cache_seqlens [batch] int32,
    weights [batch, s_next, h_idx] fp32."""
    name: str
    q_idx: torch.Tensor
    k_cache: torch.Tensor
    block_table: torch.Tensor
    cache_seqlens: torch.Tensor
    weights: torch.Tensor
    topk: int
    page: int = PAGE


def indexer_paged_case(seed: int, batch: int, s_next: int, lo: int, hi: int, h_idx: int = H_IDX,
                       d_idx: int = D_IDX, topk: int = TOPK, page: int = PAGE, spare_pages: int = 16,
                       poison: bool = True, name: str = "") -> IndexerPagedCase:
    """Request b holds L_b ~ U[lo, hi] positions; its s_next MTP query rows
    are the last s_next positions.  The page pool holds sum(ceil(L_b / page))
    + spare_pages pages in a random order (the block table is a random
    permutation); with ``poison`` every slot past a request's length, and
    every spare page, is NaN."""
    g = _gen(seed * 104729 + 7)
    lens = torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64)
    n_pages = [max(1, int(math.ceil(int(L) / page))) for L in lens]
    num_blocks = sum(n_pages) + spare_pages
    max_blocks = max(n_pages)
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    block_table = torch.zeros((batch, max_blocks), dtype=torch.int32)
    off = 0
    for b in range(batch):
        block_table[b, : n_pages[b]] = perm[off: off + n_pages[b]]
        off += n_pages[b]
    q = randn_bf16(g, (batch, s_next, h_idx, d_idx))
    k_cache = randn_bf16(g, (num_blocks, page, d_idx))
    w = indexer_weights(g, batch * s_next, h_idx, d_idx).view(batch, s_next, h_idx)
    if poison:
        keep = torch.zeros(num_blocks * page, dtype=torch.bool)
        for b in range(batch):
            pos = torch.arange(int(lens[b]), dtype=torch.int64)
            keep[block_table[b, pos // page].to(torch.int64) * page + pos % page] = True
        k_cache.view(-1, d_idx)[~keep] = float("nan")
    return IndexerPagedCase(name or f"indexer_paged_b{batch}_s{s_next}", q, k_cache, block_table,
                            lens.to(torch.int32), w, topk, page)
