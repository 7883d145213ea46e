"""Pins of the float64 oracle against facts that do not come from the oracle.

Each pin checks the oracle against something fixed by the mathematics or
by a library routine on an independent formulation:

* a dense multiplicity-matrix formulation (scores over every KV row, log
  of the per-row count added as a bias) through torch.logsumexp/softmax;
* dense causal attention through torch's scaled_dot_product_attention when
  every causal position is listed (the short-prefill case where top-k covers
  all causal positions, "feat: add XTuner TileLang sparse MLA backend",
  Summary: short prefill keeps DSA index production);
* invariance to index order and to -1 padding (the TileLang page,
  Validation: -1-padded index lists);
* closed forms: one valid entry, zero query, a duplicated entry, all masked,
  two entries, value rows of ones;
* the packed and paged variants against dense causal attention per
  sequence, a physical shuffle of the page pool and a linearised cache.

The mutation tests at the end plant plausible mistakes in a copy of the
oracle and check that at least one pin fails for each.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp as sp_logsumexp

import mla_inputs as mi
from oracle import sparse_mla_oracle as orc

D = 576
DV = 512
RT, AT = 1e-10, 1e-12


def _qkv(seed, s_q, s_kv, h):
    g = mi._gen(seed)
    return mi.randn_bf16(g, (s_q, h, D)), mi.randn_bf16(g, (s_kv, D))


def _close(a, b, rtol=RT, atol=AT):
    np.testing.assert_allclose(np.asarray(a), np.asarray(b), rtol=rtol, atol=atol)


# ---------------------------------------------------------------------------
# pins (plain functions so the mutation tests can re-run them)
# ---------------------------------------------------------------------------

def dense_count_reference(q, kv, idx, scale, dv):
    """Attention over all KV rows with log(multiplicity) as a bias."""
    qf, kf = q.double(), kv.double()
    s_q, s_kv = q.shape[0], kv.shape[0]
    count = torch.zeros(s_q, s_kv, dtype=torch.float64)
    for t in range(s_q):
        for v in idx[t].tolist():
            if 0 <= v < s_kv:
                count[t, v] += 1.0
    scores = scale * torch.einsum("thd,kd->thk", qf, kf)
    logits = scores + torch.log(count)[:, None, :]
    lse = torch.logsumexp(logits, dim=-1)
    w = torch.softmax(logits, dim=-1)
    out = w @ kf[:, :dv]
    empty = count.sum(1) == 0
    out[empty] = 0.0
    lse[empty] = -math.inf
    return out.numpy(), lse.numpy()


def pin_bruteforce_multiplicity():
    s_q, s_kv, h, topk = 7, 11, 3, 9
    q, kv = _qkv(11, s_q, s_kv, h)
    g = mi._gen(12)
    idx = torch.randint(-3, s_kv + 3, (s_q, topk), generator=g, dtype=torch.int32)
    idx[0] = -1                               # all masked
    idx[1, :] = torch.tensor([4, 4, 4, -1, 2, 2, 20, -5, -1], dtype=torch.int32)
    idx[2, :] = 3                             # one row nine times
    scale = 0.0417
    out, lse = orc.sparse_mla_fwd(q, kv, idx, scale, DV)
    ref_out, ref_lse = dense_count_reference(q, kv, idx, scale, DV)
    _close(out, ref_out)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    _close(lse[fin], ref_lse[fin])


def pin_dense_causal_sdpa():
    s, h, topk = 40, 4, 48
    q, kv = _qkv(21, s, s, h)
    g = mi._gen(22)
    idx = torch.full((s, topk), -1, dtype=torch.int32)
    for t in range(s):
        idx[t, : t + 1] = torch.randperm(t + 1, generator=g).to(torch.int32)
    idx = mi.scatter_padding(mi._gen(23), idx)
    scale = 1.0 / math.sqrt(D)
    out, lse = orc.sparse_mla_fwd(q, kv, idx, scale, DV)
    qq = q.double().permute(1, 0, 2)[None]                  # [1,h,s,D]
    kk = kv.double()[None, None].expand(1, h, s, D)
    vv = kv.double()[:, :DV][None, None].expand(1, h, s, DV)
    ref = F.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=scale)
    _close(out, ref[0].permute(1, 0, 2).numpy(), rtol=1e-9, atol=1e-11)
    sc = scale * np.einsum("thd,kd->thk", q.double().numpy(), kv.double().numpy())
    causal = np.tril(np.ones((s, s), dtype=bool))
    sc = np.where(causal[:, None, :], sc, -np.inf)
    _close(lse, sp_logsumexp(sc, axis=-1), rtol=1e-11, atol=1e-11)


def pin_order_and_padding_invariance():
    s_q, s_kv, h, topk = 6, 50, 2, 32
    q, kv = _qkv(31, s_q, s_kv, h)
    idx = mi.prefill_indices(32, s_q, s_kv, topk)
    idx[:, :] = torch.where(idx >= 0, idx + 20, idx)        # rows 20..
    base_o, base_l = orc.sparse_mla_fwd(q, kv, idx, 0.05, DV)
    perm = mi.scatter_padding(mi._gen(33), idx)
    o, l = orc.sparse_mla_fwd(q, kv, perm, 0.05, DV)
    _close(o, base_o)
    _close(l, base_l)
    wide = torch.full((s_q, topk * 3), -1, dtype=torch.int32)
    g = mi._gen(34)
    for t in range(s_q):
        pos = torch.randperm(topk * 3, generator=g)[:topk].sort().values
        wide[t, pos] = idx[t]
    o, l = orc.sparse_mla_fwd(q, kv, wide, 0.05, DV)
    _close(o, base_o)
    _close(l, base_l)


def pin_single_entry():
    q, kv = _qkv(41, 3, 9, 5)
    idx = torch.full((3, 16), -1, dtype=torch.int32)
    idx[0, 7] = 4
    idx[1, 0] = 8
    idx[2, 15] = 0
    scale = 0.3
    out, lse = orc.sparse_mla_fwd(q, kv, idx, scale, DV)
    for t, r in ((0, 4), (1, 8), (2, 0)):
        assert np.array_equal(out[t], np.broadcast_to(kv[r, :DV].double().numpy(), out[t].shape))
        for hh in range(5):
            exact = scale * math.fsum(float(a) * float(b) for a, b in
                                      zip(q[t, hh].double().tolist(), kv[r].double().tolist()))
            assert abs(lse[t, hh] - exact) <= 1e-12 * max(1.0, abs(exact))


def pin_zero_query():
    _, kv = _qkv(51, 1, 30, 1)
    q = torch.zeros(2, 3, D, dtype=torch.bfloat16)
    idx = torch.full((2, 8), -1, dtype=torch.int32)
    idx[0, :5] = torch.tensor([1, 3, 5, 7, 9])
    idx[1, :3] = torch.tensor([29, 0, 14])
    out, lse = orc.sparse_mla_fwd(q, kv, idx, 1.0, DV)
    for t, rows in ((0, [1, 3, 5, 7, 9]), (1, [29, 0, 14])):
        mean = kv[rows, :DV].double().mean(0).numpy()
        _close(out[t], np.broadcast_to(mean, out[t].shape))
        _close(lse[t], np.full(3, math.log(len(rows))), rtol=0, atol=1e-15)


def pin_duplicates_two_rows():
    q, kv = _qkv(61, 1, 4, 2)
    scale = 0.07
    for k in (1, 2, 5):
        idx = torch.full((1, 8), -1, dtype=torch.int32)
        idx[0, :k] = 1
        idx[0, k] = 3
        out, lse = orc.sparse_mla_fwd(q, kv, idx, scale, DV)
        for hh in range(2):
            s1 = scale * float(q[0, hh].double() @ kv[1].double())
            s3 = scale * float(q[0, hh].double() @ kv[3].double())
            z = k * math.exp(s1) + math.exp(s3)
            exp_out = (k * math.exp(s1) * kv[1, :DV].double() + math.exp(s3) * kv[3, :DV].double()) / z
            _close(out[0, hh], exp_out.numpy())
            assert abs(lse[0, hh] - math.log(z)) < 1e-12


def pin_all_masked():
    q, kv = _qkv(71, 2, 5, 3)
    idx = torch.tensor([[-1, -1, 5, 6], [-7, 100, -1, -1]], dtype=torch.int32)
    out, lse = orc.sparse_mla_fwd(q, kv, idx, 0.1, DV)
    assert np.all(out == 0.0) and not np.any(np.signbit(out))
    assert np.all(np.isneginf(lse))


def pin_unit_values_normalise():
    q, kv = _qkv(81, 4, 20, 3)
    kv = kv.clone()
    kv[:, :DV] = 1.0
    idx = mi.prefill_indices(82, 4, 20, 16)
    idx = torch.where(idx >= 0, idx + 10, idx)
    out, lse = orc.sparse_mla_fwd(q, kv, idx, 0.9, DV)
    _close(out, np.ones_like(out), rtol=0, atol=1e-14)
    assert np.all(np.isfinite(lse))


PINS = [pin_bruteforce_multiplicity, pin_dense_causal_sdpa, pin_order_and_padding_invariance,
        pin_single_entry, pin_zero_query, pin_duplicates_two_rows, pin_all_masked,
        pin_unit_values_normalise]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_fwd_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# packed prefill
# ---------------------------------------------------------------------------

def test_varlen_dense_causal_per_sequence():
    seqlens, h, topk = [17, 5, 30, 1], 3, 32
    case = mi.varlen_case(91, seqlens, h, topk=topk)
    out, lse = orc.sparse_mla_fwd_varlen(case.q, case.kv, case.indices, case.cu_seqlens_q,
                                         case.cu_seqlens_kv, case.sm_scale, DV)
    cu = case.cu_seqlens_q.tolist()
    for b, L in enumerate(seqlens):
        a = cu[b]
        qq = case.q[a:a + L].double().permute(1, 0, 2)[None]
        kk = case.kv[a:a + L].double()[None, None].expand(1, h, L, D)
        vv = case.kv[a:a + L, :DV].double()[None, None].expand(1, h, L, DV)
        ref = F.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=case.sm_scale)
        _close(out[a:a + L], ref[0].permute(1, 0, 2).numpy(), rtol=1e-9, atol=1e-11)
        o2, l2 = orc.sparse_mla_fwd(case.q[a:a + L], case.kv[a:a + L], case.indices[a:a + L],
                                    case.sm_scale, DV)
        _close(out[a:a + L], o2)
        _close(lse[a:a + L], l2)


def test_varlen_local_indices_past_sequence_are_masked():
    case = mi.varlen_case(92, [6, 9], 2, topk=12)
    idx = case.indices.clone()
    idx[0, 1] = 6          # inside the packed tensor, outside sequence 0
    idx[7, 11] = 9         # one past sequence 1
    o, l = orc.sparse_mla_fwd_varlen(case.q, case.kv, idx, case.cu_seqlens_q,
                                     case.cu_seqlens_kv, case.sm_scale, DV)
    o0, l0 = orc.sparse_mla_fwd_varlen(case.q, case.kv, case.indices, case.cu_seqlens_q,
                                       case.cu_seqlens_kv, case.sm_scale, DV)
    _close(o, o0)
    _close(l, l0)


# ---------------------------------------------------------------------------
# paged decode
# ---------------------------------------------------------------------------

def _small_decode(seed=101, topk=64):
    return mi.decode_case(seed, batch=3, s_next=2, h_q=4, lo=70, hi=200, topk=topk,
                          page=16, spare_pages=5)


def test_decode_matches_linearised_cache():
    c = _small_decode()
    out, lse = orc.sparse_mla_decode(c.q, c.kv_cache, c.block_table, c.cache_seqlens,
                                     c.indices, c.sm_scale, c.page_size, DV)
    out = out.reshape(c.batch, c.s_next, c.h_q, DV)
    lse = lse.reshape(c.batch, c.s_next, c.h_q)
    for b in range(c.batch):
        L = int(c.cache_seqlens[b])
        pages = c.block_table[b, : (L + c.page_size - 1) // c.page_size].long()
        lin = c.kv_cache[pages].reshape(-1, D)[:L]
        o2, l2 = orc.sparse_mla_fwd(c.q[b], lin, c.indices[b], c.sm_scale, DV)
        _close(out[b], o2)
        _close(lse[b], l2)
    assert np.all(np.isfinite(out))


def test_decode_page_shuffle_invariance():
    c = _small_decode(102)
    out, lse = orc.sparse_mla_decode(c.q, c.kv_cache, c.block_table, c.cache_seqlens,
                                     c.indices, c.sm_scale, c.page_size, DV)
    nb = c.kv_cache.shape[0]
    perm = torch.randperm(nb, generator=mi._gen(103))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    cache2 = c.kv_cache[perm]                 # new page p holds old page perm[p]
    table2 = inv[c.block_table.long()].to(torch.int32)
    o2, l2 = orc.sparse_mla_decode(c.q, cache2, table2, c.cache_seqlens, c.indices,
                                   c.sm_scale, c.page_size, DV)
    _close(o2, out)
    _close(l2, lse)


def test_decode_dense_causal_sdpa():
    batch, s_next, h, page, topk = 2, 3, 2, 16, 64
    c = mi.decode_case(104, batch, s_next, h, lo=30, hi=60, topk=topk, page=page,
                       spare_pages=2, poison=False)
    idx = torch.full_like(c.indices, -1)
    g = mi._gen(105)
    for b in range(batch):
        L = int(c.cache_seqlens[b])
        for j in range(s_next):
            n = L - s_next + j + 1
            idx[b, j, :n] = torch.randperm(n, generator=g).to(torch.int32)
    out, _ = orc.sparse_mla_decode(c.q, c.kv_cache, c.block_table, c.cache_seqlens, idx,
                                   c.sm_scale, page, DV)
    out = out.reshape(batch, s_next, h, DV)
    for b in range(batch):
        L = int(c.cache_seqlens[b])
        pages = c.block_table[b, : (L + page - 1) // page].long()
        lin = c.kv_cache[pages].reshape(-1, D)[:L].double()
        mask = torch.zeros(s_next, L, dtype=torch.bool)
        for j in range(s_next):
            mask[j, : L - s_next + j + 1] = True
        qq = c.q[b].double().permute(1, 0, 2)[None]
        kk = lin[None, None].expand(1, h, L, D)
        vv = lin[:, :DV][None, None].expand(1, h, L, DV)
        ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=c.sm_scale)
        _close(out[b], ref[0].permute(1, 0, 2).numpy(), rtol=1e-9, atol=1e-11)


def test_decode_poisoned_slots_never_read():
    c = _small_decode(106)
    out, lse = orc.sparse_mla_decode(c.q, c.kv_cache, c.block_table, c.cache_seqlens,
                                     c.indices, c.sm_scale, c.page_size, DV)
    assert torch.isnan(c.kv_cache.float()).any()
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_decode_invalid_pages_are_masked():
    """Masking beyond -1 on the paged layout: an index whose page lies past
    the block table's width, or whose table entry falls outside
    [0, num_blocks), counts as masked.  Pinned against the plain forward over
    each request's linearised cache with those entries replaced by -1 on the
    host (placeholder rows of zeros where a page is missing)."""
    c = _small_decode(107)
    nb, page = c.kv_cache.shape[0], c.page_size
    width = 6                                           # pages 0..5: positions >= 96 have no page
    bt = c.block_table[:, :width].clone()
    bt[0, 1] = -5                                       # outside the pool, below
    bt[1, 2] = nb + 3                                   # outside the pool, above
    out, lse = orc.sparse_mla_decode(c.q, c.kv_cache, bt, c.cache_seqlens, c.indices, c.sm_scale, page, DV)
    out = out.reshape(c.batch, c.s_next, c.h_q, DV)
    lse = lse.reshape(c.batch, c.s_next, c.h_q)
    masked_any = False
    for b in range(c.batch):
        L = int(c.cache_seqlens[b])
        lin = torch.zeros((L, D), dtype=c.kv_cache.dtype)
        good = torch.zeros(L, dtype=torch.bool)
        for pg in range(min(width, (L + page - 1) // page)):
            e = int(bt[b, pg])
            if 0 <= e < nb:
                n = min(page, L - pg * page)
                lin[pg * page: pg * page + n] = c.kv_cache[e, :n]
                good[pg * page: pg * page + n] = True
        idx = c.indices[b].clone()
        inside = (idx >= 0) & (idx < L)
        bad = inside & ~good[idx.clamp(0, L - 1).long()]
        masked_any |= bool(bad.any())
        idx[bad] = -1
        o2, l2 = orc.sparse_mla_fwd(c.q[b], lin, idx, c.sm_scale, DV)
        _close(out[b], o2)
        _close(lse[b], l2)
    assert masked_any


def test_valid_count_bruteforce():
    idx = torch.tensor([[-1, 0, 3, 3, 9], [10, -2, -1, -1, 4]], dtype=torch.int32)
    assert orc.valid_count_dense(idx, 10).tolist() == [4, 1]


def test_valid_count_varlen_by_hand():
    """Two sequences of 3 and 5 positions; local indices only count inside
    their own sequence (counts written out by hand)."""
    cu_q = torch.tensor([0, 2, 4], dtype=torch.int32)
    cu_k = torch.tensor([0, 3, 8], dtype=torch.int32)
    idx = torch.tensor([[0, 2, 3, -1],      # seq 0: 3 is past its 3 positions -> 2
                        [2, 2, -2, 1],      # seq 0: duplicates count twice -> 3
                        [4, 5, 7, 0],       # seq 1 (5 positions): 5 and 7 past -> 2
                        [-1, -1, -1, -1]], dtype=torch.int32)
    assert orc.valid_count_varlen(idx, cu_q, cu_k).tolist() == [2, 3, 2, 0]


def test_valid_count_paged_by_hand():
    """Pages of 4 slots, a pool of 5 pages, two requests with a table two
    pages wide: request 0 has pages [3, -1] and 7 tokens; request 1 has
    pages [9, 0] (9 outside the pool) and 8 tokens."""
    table = torch.tensor([[3, -1], [9, 0]], dtype=torch.int32)
    lens = torch.tensor([7, 8], dtype=torch.int32)
    idx = torch.tensor([[[0, 3, 4, 6], [6, 7, 8, -1]],      # r0: page 1 is -1 -> 2 ; 7, 8 past the length -> 0
                        [[0, 4, 7, 8], [5, 5, -3, 3]]],     # r1: page 0 is 9 -> only 4, 7 -> 2 ; 5, 5 -> 2
                       dtype=torch.int32)
    assert orc.valid_count_paged(idx, table, lens, 4, 5).tolist() == [2, 0, 2, 2]


# ---------------------------------------------------------------------------
# mutation tests: each planted mistake must fail at least one pin
# ---------------------------------------------------------------------------

def _attend_wrong_value_slice(q_t, rows, sm_scale, d_v):
    r2 = rows.copy()
    r2[:, :d_v] = rows[:, rows.shape[1] - d_v:]
    return _TRUE_ATTEND(q_t, r2, sm_scale, d_v)


def _attend_no_scale(q_t, rows, sm_scale, d_v):
    return _TRUE_ATTEND(q_t, rows, 1.0, d_v)


def _attend_log2(q_t, rows, sm_scale, d_v):
    o, l = _TRUE_ATTEND(q_t, rows, sm_scale, d_v)
    return o, l / math.log(2.0)


def _attend_unique(q_t, rows, sm_scale, d_v):
    return _TRUE_ATTEND(q_t, np.unique(rows, axis=0) if rows.shape[0] else rows, sm_scale, d_v)


def _attend_drop_rope(q_t, rows, sm_scale, d_v):
    r2 = rows.copy()
    r2[:, d_v:] = 0.0
    return _TRUE_ATTEND(q_t, r2, sm_scale, d_v)


def _attend_lse_without_max(q_t, rows, sm_scale, d_v):
    o, l = _TRUE_ATTEND(q_t, rows, sm_scale, d_v)
    if rows.shape[0] == 0:
        return o, l
    s = sm_scale * (q_t @ rows.T)
    return o, l - s.max(axis=1)


def _attend_sign(q_t, rows, sm_scale, d_v):
    return _TRUE_ATTEND(-q_t, rows, sm_scale, d_v)


def _rows_dense_minus_one_wraps(idx_t, s_kv):
    v = idx_t[(idx_t >= -1) & (idx_t < s_kv)]
    return np.where(v < 0, s_kv - 1, v)


_TRUE_ATTEND = orc.attend
MUTANTS = [("attend", _attend_wrong_value_slice), ("attend", _attend_no_scale),
           ("attend", _attend_log2), ("attend", _attend_unique),
           ("attend", _attend_drop_rope), ("attend", _attend_lse_without_max),
           ("attend", _attend_sign), ("rows_dense", _rows_dense_minus_one_wraps)]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, name, fn):
    monkeypatch.setattr(orc, name, fn)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"no pin caught the planted mistake {fn.__name__}"


# ---------------------------------------------------------------------------
# indices-free causal mode
# ---------------------------------------------------------------------------

def _bottom_right_sdpa(q, kv, scale):
    """float64 attention of the s_q queries, taken as the last s_q of s_kv
    positions, over every KV position at or before their own, through
    torch's scaled_dot_product_attention with an explicit mask; plus the LSE
    from scipy's logsumexp over the same mask."""
    s_q, h = q.shape[0], q.shape[1]
    s_kv = kv.shape[0]
    mask = np.arange(s_kv)[None, :] <= (np.arange(s_q) + s_kv - s_q)[:, None]      # [s_q, s_kv]
    qq = q.double().permute(1, 0, 2)[None]
    kk = kv.double()[None, None].expand(1, h, s_kv, D)
    vv = kv.double()[:, :DV][None, None].expand(1, h, s_kv, DV)
    ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=torch.from_numpy(mask), scale=scale)
    sc = scale * np.einsum("thd,kd->thk", q.double().numpy(), kv.double().numpy())
    sc = np.where(mask[:, None, :], sc, -np.inf)
    return ref[0].permute(1, 0, 2).numpy(), sp_logsumexp(sc, axis=-1), mask


def pin_causal_square():
    s, h = 40, 4
    q, kv = _qkv(31, s, s, h)
    scale = 1.0 / math.sqrt(D)
    out, lse = orc.causal_mla_fwd(q, kv, scale, DV)
    qq = q.double().permute(1, 0, 2)[None]
    kk = kv.double()[None, None].expand(1, h, s, D)
    vv = kv.double()[:, :DV][None, None].expand(1, h, s, DV)
    ref = F.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=scale)
    _close(out, ref[0].permute(1, 0, 2).numpy(), rtol=1e-9, atol=1e-11)
    ref_o, ref_l, _ = _bottom_right_sdpa(q, kv, scale)
    _close(lse, ref_l, rtol=1e-11, atol=1e-11)


def pin_causal_queries_are_the_last_positions():
    s_q, s_kv, h = 13, 50, 3
    q, kv = _qkv(32, s_q, s_kv, h)
    scale = 0.05
    out, lse = orc.causal_mla_fwd(q, kv, scale, DV)
    ref_o, ref_l, _ = _bottom_right_sdpa(q, kv, scale)
    _close(out, ref_o, rtol=1e-9, atol=1e-11)
    _close(lse, ref_l, rtol=1e-11, atol=1e-11)


def pin_causal_queries_before_the_first_position():
    """More queries than KV rows: the first s_q - s_kv attend to nothing."""
    s_q, s_kv, h = 10, 4, 2
    q, kv = _qkv(33, s_q, s_kv, h)
    out, lse = orc.causal_mla_fwd(q, kv, 0.07, DV)
    assert np.all(out[:6] == 0.0) and np.all(np.isneginf(lse[:6]))
    ref_o, ref_l, _ = _bottom_right_sdpa(q[6:], kv, 0.07)
    _close(out[6:], ref_o, rtol=1e-9, atol=1e-11)
    _close(lse[6:], ref_l, rtol=1e-11, atol=1e-11)


def pin_causal_equals_full_causal_lists():
    """The mode is the sparse forward given every causal position as its list."""
    s_q, s_kv, h = 9, 20, 2
    q, kv = _qkv(34, s_q, s_kv, h)
    idx = torch.full((s_q, s_kv), -1, dtype=torch.int32)
    for t in range(s_q):
        idx[t, : t + s_kv - s_q + 1] = torch.arange(t + s_kv - s_q + 1, dtype=torch.int32)
    o1, l1 = orc.causal_mla_fwd(q, kv, 0.04, DV)
    o2, l2 = orc.sparse_mla_fwd(q, kv, idx, 0.04, DV)
    _close(o1, o2, rtol=1e-13, atol=1e-14)
    _close(l1, l2, rtol=1e-13, atol=1e-14)


CAUSAL_PINS = [pin_causal_square, pin_causal_queries_are_the_last_positions,
               pin_causal_queries_before_the_first_position, pin_causal_equals_full_causal_lists]


@pytest.mark.parametrize("pin", CAUSAL_PINS, ids=[p.__name__ for p in CAUSAL_PINS])
def test_causal_pin(pin):
    pin()


def _causal_off_by_one(q, kv, sm_scale, d_v=512, tokens=None):
    s_q, s_kv = q.shape[0], kv.shape[0]
    outs, lses = [], []
    for t in range(s_q):
        r = np.arange(0, max(0, min(t + s_kv - s_q, s_kv)), dtype=np.int64)    # position t itself left out
        o, l = orc.attend(orc._f64(q[t]), orc._gather(kv, r), sm_scale, d_v)
        outs.append(o)
        lses.append(l)
    return orc._stack(outs, lses, q.shape[1], d_v)


def _causal_top_left(q, kv, sm_scale, d_v=512, tokens=None):
    s_q, s_kv = q.shape[0], kv.shape[0]
    outs, lses = [], []
    for t in range(s_q):
        r = np.arange(0, min(t + 1, s_kv), dtype=np.int64)                        # queries taken as the first positions
        o, l = orc.attend(orc._f64(q[t]), orc._gather(kv, r), sm_scale, d_v)
        outs.append(o)
        lses.append(l)
    return orc._stack(outs, lses, q.shape[1], d_v)


_TRUE_CAUSAL = orc.causal_mla_fwd


def _causal_unscaled(q, kv, sm_scale, d_v=512, tokens=None):
    return _TRUE_CAUSAL(q, kv, 1.0, d_v, tokens)


@pytest.mark.parametrize("fn", [_causal_off_by_one, _causal_top_left, _causal_unscaled],
                         ids=lambda f: f.__name__)
def test_causal_pins_catch_planted_mistake(monkeypatch, fn):
    monkeypatch.setattr(orc, "causal_mla_fwd", fn)
    failed = 0
    for pin in CAUSAL_PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"no pin caught the planted mistake {fn.__name__}"


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------

def _autograd_reference(q, kv, idx, scale, dout):
    """dq, dkv by torch autograd (float64) through a dense formulation of the
    forward: scores over every kv row plus log(multiplicity of the row in the
    token's list), softmax, times kv[:, :512]; loss = sum(out * dout) over the
    tokens that have a valid entry."""
    s_q, h = q.shape[0], q.shape[1]
    s_kv = kv.shape[0]
    qv = q.double().clone().requires_grad_(True)
    kvv = kv.double().clone().requires_grad_(True)
    count = torch.zeros((s_q, s_kv), dtype=torch.float64)
    for t in range(s_q):
        for i in idx[t].tolist():
            if 0 <= i < s_kv:
                count[t, i] += 1
    live = count.sum(1) > 0
    scores = scale * torch.einsum("thd,kd->thk", qv, kvv) + torch.log(count)[:, None, :]
    w = torch.softmax(scores[live], dim=-1)
    out = w @ kvv[:, :DV]
    (out * dout.double()[live]).sum().backward()
    return qv.grad.numpy(), kvv.grad.numpy()


def pin_bwd_autograd():
    s_q, s_kv, h, topk = 9, 23, 3, 12
    q, kv = _qkv(41, s_q, s_kv, h)
    g = mi._gen(42)
    idx = torch.randint(-2, s_kv + 2, (s_q, topk), generator=g, dtype=torch.int32)
    idx[0] = -1                                   # no valid entry: zero gradient
    idx[1, :4] = torch.tensor([5, 5, 5, 7], dtype=torch.int32)   # multiplicity
    dout = torch.randn((s_q, h, DV), generator=g, dtype=torch.float64)
    scale = 0.0417
    dq, dkv = orc.sparse_mla_bwd(q, kv, idx, scale, dout, DV)
    rq, rkv = _autograd_reference(q, kv, idx, scale, dout)
    _close(dq, rq, rtol=1e-9, atol=1e-12)
    _close(dkv, rkv, rtol=1e-9, atol=1e-12)
    assert np.all(dq[0] == 0.0)


def pin_bwd_finite_differences():
    """Central differences of L = sum(out * dout) through the float64 forward
    oracle, along random directions in q and in kv."""
    s_q, s_kv, h, topk = 3, 7, 2, 6
    q, kv = _qkv(43, s_q, s_kv, h)
    q, kv = q.double(), kv.double()
    g = mi._gen(44)
    idx = torch.randint(0, s_kv, (s_q, topk), generator=g, dtype=torch.int32)
    dout = torch.randn((s_q, h, DV), generator=g, dtype=torch.float64)
    scale = 0.05
    dq, dkv = orc.sparse_mla_bwd(q, kv, idx, scale, dout, DV)

    def loss(qq, kk):
        out, _ = orc.sparse_mla_fwd(qq, kk, idx, scale, DV)
        return float((out * dout.numpy()).sum())
    eps = 1e-5
    for _ in range(3):
        dqd = torch.randn(q.shape, generator=g, dtype=torch.float64)
        fd = (loss(q + eps * dqd, kv) - loss(q - eps * dqd, kv)) / (2 * eps)
        assert abs(fd - float((dq * dqd.numpy()).sum())) <= 1e-6 * (1 + abs(fd)), "dq vs finite differences"
        dkd = torch.randn(kv.shape, generator=g, dtype=torch.float64)
        fd = (loss(q, kv + eps * dkd) - loss(q, kv - eps * dkd)) / (2 * eps)
        assert abs(fd - float((dkv * dkd.numpy()).sum())) <= 1e-6 * (1 + abs(fd)), "dkv vs finite differences"


BWD_PINS = [pin_bwd_autograd, pin_bwd_finite_differences]


@pytest.mark.parametrize("pin", BWD_PINS, ids=[p.__name__ for p in BWD_PINS])
def test_bwd_pin(pin):
    pin()


_TRUE_BWD = orc.sparse_mla_bwd


def _bwd_variant(drop_d=False, unscaled_dq=False, v_into_rope=False, no_multiplicity=False):
    def f(q, kv, indices, sm_scale, dout, d_v=512):
        s_q, h = q.shape[0], q.shape[1]
        kv2 = kv.reshape(kv.shape[0], -1)
        s_kv, d_qk = kv2.shape
        idx = orc._i64(indices).reshape(s_q, -1)
        q64, do64 = orc._f64(q), orc._f64(dout)
        dq = np.zeros((s_q, h, d_qk))
        dkv = np.zeros((s_kv, d_qk))
        for t in range(s_q):
            r = orc.rows_dense(idx[t], s_kv)
            if r.size == 0:
                continue
            K = orc._gather(kv2, r)
            V = K if v_into_rope else K[:, :d_v]
            s = sm_scale * (q64[t] @ K.T)
            P = np.exp(s - s.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            dP = do64[t] @ K[:, :d_v].T
            D = 0.0 if drop_d else (do64[t] * (P @ K[:, :d_v])).sum(axis=1, keepdims=True)
            dS = P * (dP - D)
            dq[t] = (1.0 if unscaled_dq else sm_scale) * (dS @ K)
            dk = sm_scale * (dS.T @ q64[t])
            dv = P.T @ do64[t]
            if v_into_rope:
                dv = np.concatenate([dv, dv[:, :d_qk - d_v]], axis=1)
                dk = dk + dv
            else:
                dk[:, :d_v] += dv
            if no_multiplicity:
                dkv[r] += dk
            else:
                np.add.at(dkv, r, dk)
        return dq, dkv
    return f


BWD_MUTANTS = [("drop_d", _bwd_variant(drop_d=True)), ("unscaled_dq", _bwd_variant(unscaled_dq=True)),
               ("v_into_rope", _bwd_variant(v_into_rope=True)), ("no_multiplicity", _bwd_variant(no_multiplicity=True))]


@pytest.mark.parametrize("name,fn", BWD_MUTANTS, ids=[m[0] for m in BWD_MUTANTS])
def test_bwd_pins_catch_planted_mistake(monkeypatch, name, fn):
    monkeypatch.setattr(orc, "sparse_mla_bwd", fn)
    failed = 0
    for pin in BWD_PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"no pin caught the planted mistake {name}"


def test_bwd_varlen_autograd_per_sequence():
    """Packed backward: per sequence, torch autograd on the sequence's own
    slice with its local indices; kv rows of other sequences get nothing
    from it."""
    seqlens, h, topk = [9, 3, 14], 2, 10
    case = mi.varlen_case(47, seqlens, h, topk=topk)
    g = mi._gen(48)
    dout = torch.randn((sum(seqlens), h, DV), generator=g, dtype=torch.float64)
    dq, dkv = orc.sparse_mla_bwd_varlen(case.q, case.kv, case.indices, case.cu_seqlens_q, case.cu_seqlens_kv,
                                        case.sm_scale, dout, DV)
    cu, ck = case.cu_seqlens_q.tolist(), case.cu_seqlens_kv.tolist()
    for b in range(len(seqlens)):
        a, e = cu[b], cu[b + 1]
        rq, rkv = _autograd_reference(case.q[a:e], case.kv[ck[b]:ck[b + 1]], case.indices[a:e], case.sm_scale,
                                      dout[a:e])
        _close(dq[a:e], rq, rtol=1e-9, atol=1e-12)
        _close(dkv[ck[b]:ck[b + 1]], rkv, rtol=1e-9, atol=1e-12)


def test_bwd_variant_without_mistakes_passes():
    """The mutation harness itself is faithful: with no mistake planted it
    reproduces the oracle."""
    s_q, s_kv, h = 5, 11, 2
    q, kv = _qkv(45, s_q, s_kv, h)
    g = mi._gen(46)
    idx = torch.randint(-1, s_kv, (s_q, 8), generator=g, dtype=torch.int32)
    dout = torch.randn((s_q, h, DV), generator=g, dtype=torch.float64)
    a = _TRUE_BWD(q, kv, idx, 0.03, dout, DV)
    b = _bwd_variant()(q, kv, idx, 0.03, dout, DV)
    _close(a[0], b[0], rtol=1e-12, atol=1e-14)
    _close(a[1], b[1], rtol=1e-12, atol=1e-14)


def test_generator_valid_row_counts():
    """Valid-entry totals of the workloads equal their closed forms:
    sum_i min(i+1, 2048) per sequence; 96*2048 for the decode batch."""
    def closed(L, k=2048):
        return sum(min(i + 1, k) for i in range(L))
    assert int((mi.prefill_indices(1001, 64, 64) >= 0).sum()) == closed(64) == 2080
    assert int((mi.prefill_indices(1002, 2119, 2119) >= 0).sum()) == closed(2119) == 2243584
    assert closed(8192) == 14681088
    assert sum(closed(L) for L in mi.VARLEN_C4) == 24121344
    idx, cu, _ = mi.varlen_indices(7, [300, 5, 2100], topk=2048)
    assert int((idx >= 0).sum()) == closed(300) + closed(5) + closed(2100)
    assert cu.tolist() == [0, 300, 305, 2405]
