"""Pins of the float64 DSA indexer / top-k oracle against facts that do not
come from the oracle:

* a worked example in small integers whose scores and lists are computed
  by hand (the scores are exact in float64);
* the ReLU's zero floor: a key anti-aligned with every head's query scores
  exactly 0 whatever the weights;
* positive homogeneity and additivity of the scores in the weights, and
  homogeneity in the queries;
* the selection against brute-force properties on tied integer scores
  (every selected score >= every unselected one, ties at the boundary go to
  the smaller positions, increasing order, -1 padding) and against
  torch.topk on distinct scores;
* causal visibility in closed form (square, cached prefix, more queries than
  positions) and the short-row identity lists;
* the packed form against the dense form per sequence;
* the link to the forward: when every row is short, the sparse forward over
  these lists equals the indices-free causal forward (itself pinned to
  torch's scaled_dot_product_attention).

The mutation tests at the end plant plausible mistakes in the oracle and
check that at least one pin fails for each.
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi
from oracle import dsa_indexer_oracle as ido
from oracle import sparse_mla_oracle as orc


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def _worked():
    """Two heads of width 2, three KV positions and two queries, the last two
    of the three positions (query 0 sees positions 0, 1; query 1 sees 0, 1,
    2)."""
    q = torch.tensor([[[0.0, 1.0], [1.0, 1.0]],      # query 0
                      [[1.0, 0.0], [0.0, 1.0]]])     # query 1
    k = torch.tensor([[3.0, -1.0], [-2.0, 4.0], [1.0, 1.0]])
    w = torch.tensor([[1.0, -1.0], [1.0, 2.0]])
    return q, k, w


def pin_worked_example_scores():
    q, k, w = _worked()
    s = ido.indexer_scores(q, k, w)
    # query 0: position 0: head0 relu(-1)=0, head1 relu(3-1)=2 -> 1*0 - 1*2 = -2
    #          position 1: head0 relu(4)=4,  head1 relu(-2+4)=2 -> 4 - 2 = 2
    # query 1: position 0: relu(3)=3, relu(-1)=0 -> 3
    #          position 1: relu(-2)=0, relu(4)=4 -> 2*4 = 8
    #          position 2: relu(1)=1, relu(1)=1 -> 1 + 2 = 3
    expect = np.array([[-2.0, 2.0, -np.inf], [3.0, 8.0, 3.0]])
    np.testing.assert_array_equal(s, expect)


def pin_worked_example_lists():
    q, k, w = _worked()
    # topk 1: query 0 -> position 1 (2 > -2); query 1 -> position 1 (8)
    np.testing.assert_array_equal(ido.dsa_indices(q, k, w, 1), [[1], [1]])
    # topk 2: query 0 sees two positions (short row: identity list);
    # query 1 keeps 8 at position 1 and the tie 3 / 3 goes to position 0
    np.testing.assert_array_equal(ido.dsa_indices(q, k, w, 2), [[0, 1], [0, 1]])
    # topk 4: every visible position, -1 padded
    np.testing.assert_array_equal(ido.dsa_indices(q, k, w, 4), [[0, 1, -1, -1], [0, 1, 2, -1]])


def pin_relu_floor():
    g = mi._gen(71)
    h, d = 5, 16
    q = torch.rand((1, h, d), generator=g) + 0.1          # every query positive
    k = torch.rand((4, d), generator=g) + 0.1
    k[2] = -k[2]                                           # anti-aligned with every head
    w = torch.randn((1, h), generator=g)
    s = ido.indexer_scores(q, k, w)
    assert s[0, 2] == 0.0
    assert np.all(np.abs(s[0, [0, 1, 3]]) > 0)


def pin_weight_homogeneity_additivity():
    c = mi.indexer_case(72, 6, 40, h_idx=8, d_idx=32)
    s = ido.indexer_scores(c.q_idx, c.k_idx, c.weights)
    s3 = ido.indexer_scores(c.q_idx, c.k_idx, c.weights.double() * 3.0)
    fin = np.isfinite(s)
    np.testing.assert_allclose(s3[fin], 3.0 * s[fin], rtol=1e-12, atol=1e-14)
    w2 = torch.randn(c.weights.shape, generator=mi._gen(73), dtype=torch.float64)
    sa = ido.indexer_scores(c.q_idx, c.k_idx, c.weights.double() + w2)
    sb = ido.indexer_scores(c.q_idx, c.k_idx, w2)
    np.testing.assert_allclose(sa[fin], s[fin] + sb[fin], rtol=1e-11, atol=1e-12)
    sq = ido.indexer_scores(c.q_idx.double() * 0.5, c.k_idx, c.weights)
    np.testing.assert_allclose(sq[fin], 0.5 * s[fin], rtol=1e-12, atol=1e-14)
    # selection is invariant to a positive scale of the weights
    np.testing.assert_array_equal(ido.dsa_indices(c.q_idx, c.k_idx, c.weights, 8),
                                  ido.dsa_indices(c.q_idx, c.k_idx, c.weights.double() * 5.0, 8))


def _check_selection(scores_row, v, topk, lst):
    """Brute-force properties of one list against scores_row[:v]."""
    lst = np.asarray(lst)
    n = min(topk, v)
    assert np.all(lst[n:] == -1)
    sel = lst[:n]
    assert np.all(sel >= 0) and np.all(sel < v)
    assert np.all(np.diff(sel) > 0), "increasing positions, no repeats"
    if v <= topk:
        np.testing.assert_array_equal(sel, np.arange(v))
        return
    chosen = np.zeros(v, dtype=bool)
    chosen[sel] = True
    sv = np.asarray(scores_row[:v], dtype=np.float64)
    lo = sv[chosen].min()
    assert sv[~chosen].max() <= lo
    # at the boundary value, the chosen positions precede the others
    tie_in = np.nonzero(chosen & (sv == lo))[0]
    tie_out = np.nonzero(~chosen & (sv == lo))[0]
    if tie_out.size:
        assert tie_in.max() < tie_out.min()


def pin_selection_properties_with_ties():
    sc = mi.tied_scores(74, 12, 60).numpy().astype(np.float64)
    lens = [0, 1, 5, 9, 10, 11, 30, 45, 59, 60, 60, 33]
    for topk in (1, 3, 10, 32, 64):
        out = ido.topk_rows(sc, lens, topk)
        for i, v in enumerate(lens):
            _check_selection(sc[i], v, topk, out[i])


def pin_selection_matches_torch_topk():
    g = mi._gen(75)
    sc = torch.randn((5, 300), generator=g, dtype=torch.float64)    # distinct almost surely
    assert all(torch.unique(sc[i]).numel() == 300 for i in range(5))
    out = ido.topk_rows(sc.numpy(), [300] * 5, 37)
    for i in range(5):
        ref = torch.sort(torch.topk(sc[i], 37).indices).values.numpy()
        np.testing.assert_array_equal(out[i], ref)


def pin_visibility_closed_forms():
    assert [ido.visible_len(t, 5, 5) for t in range(5)] == [1, 2, 3, 4, 5]
    assert [ido.visible_len(t, 3, 10) for t in range(3)] == [8, 9, 10]     # 7 cached positions
    assert [ido.visible_len(t, 6, 4) for t in range(6)] == [0, 0, 1, 2, 3, 4]   # two queries before position 0
    c = mi.indexer_case(76, 6, 4, h_idx=4, d_idx=8)
    lst = ido.dsa_indices(c.q_idx, c.k_idx, c.weights, 2)
    np.testing.assert_array_equal(lst[:2], -1)
    np.testing.assert_array_equal(lst[2], [0, -1])
    np.testing.assert_array_equal(lst[3], [0, 1])
    # rows 4 and 5 see 3 and 4 > 2 positions: scored rows with two entries
    assert (lst[4] >= 0).sum() == 2 and (lst[5] >= 0).sum() == 2


def pin_scores_selection_consistent():
    c = mi.indexer_case(77, 20, 70, h_idx=8, d_idx=32, topk=16)
    s = ido.indexer_scores(c.q_idx, c.k_idx, c.weights)
    lst = ido.dsa_indices(c.q_idx, c.k_idx, c.weights, 16)
    for t in range(20):
        v = ido.visible_len(t, 20, 70)
        assert np.all(np.isinf(s[t, v:])) and np.all(np.isfinite(s[t, :v]))
        _check_selection(s[t], v, 16, lst[t])


def pin_varlen_matches_dense_per_sequence():
    c = mi.indexer_varlen_case(78, [5, 12, 1, 9], [5, 30, 4, 9], h_idx=8, d_idx=32, topk=6)
    got = ido.dsa_indices_varlen(c.q_idx, c.k_idx, c.weights, c.cu_seqlens_q, c.cu_seqlens_kv, 6)
    gs = ido.indexer_scores_varlen(c.q_idx, c.k_idx, c.weights, c.cu_seqlens_q, c.cu_seqlens_kv)
    cq, ck = c.cu_seqlens_q.tolist(), c.cu_seqlens_kv.tolist()
    for b in range(4):
        qs, ks = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
        ref = ido.dsa_indices(c.q_idx[qs], c.k_idx[ks], c.weights[qs], 6)
        np.testing.assert_array_equal(got[qs], ref)
        rs = ido.indexer_scores(c.q_idx[qs], c.k_idx[ks], c.weights[qs])
        np.testing.assert_array_equal(gs[qs, :rs.shape[1]], rs)


def pin_short_rows_reproduce_causal_forward():
    s, h = 24, 2
    c = mi.indexer_case(79, s, s, h_idx=4, d_idx=8, topk=32)
    lst = ido.dsa_indices(c.q_idx, c.k_idx, c.weights, 32)
    g = mi._gen(80)
    q = mi.randn_bf16(g, (s, h, mi.D_QK))
    kv = mi.randn_bf16(g, (s, mi.D_QK))
    scale = mi.default_sm_scale()
    o1, l1 = orc.sparse_mla_fwd(q, kv, torch.from_numpy(lst), scale)
    o2, l2 = orc.causal_mla_fwd(q, kv, scale)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-13)


def _paged(seed, poison=True):
    return mi.indexer_paged_case(seed, 3, 5, 60, 330, h_idx=8, d_idx=32, topk=48, poison=poison)


def pin_paged_identity_table_is_dense():
    """One request whose block table is the identity: the dense oracle on the
    cache read as one row per position."""
    c = mi.indexer_paged_case(81, 1, 4, 200, 200, h_idx=8, d_idx=32, topk=40, spare_pages=0, poison=False)
    bt = torch.arange(c.block_table.shape[1], dtype=torch.int32)[None]
    got = ido.dsa_indices_paged(c.q_idx, c.k_cache, c.weights, bt, c.cache_seqlens, 40, c.page)
    k_lin = c.k_cache.reshape(-1, c.k_cache.shape[-1])[:200]
    ref = ido.dsa_indices(c.q_idx[0], k_lin, c.weights[0], 40)
    np.testing.assert_array_equal(got, ref)


def pin_paged_matches_packed_on_linearised_keys():
    c = _paged(82)
    b_n, s_next = c.q_idx.shape[0], c.q_idx.shape[1]
    lens = [int(x) for x in c.cache_seqlens]
    keys = torch.cat([torch.from_numpy(ido.linearise_keys(c.k_cache, c.block_table[b], lens[b], c.page))
                      for b in range(b_n)])
    cq = torch.arange(0, (b_n + 1) * s_next, s_next, dtype=torch.int32)
    ck = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32)
    ref = ido.dsa_indices_varlen(c.q_idx.reshape(b_n * s_next, *c.q_idx.shape[2:]), keys,
                                 c.weights.reshape(b_n * s_next, -1), cq, ck, 48)
    got = ido.dsa_indices_paged(c.q_idx, c.k_cache, c.weights, c.block_table, c.cache_seqlens, 48, c.page)
    np.testing.assert_array_equal(got, ref)


def pin_paged_page_shuffle_invariance():
    c = _paged(83)
    perm = torch.randperm(c.k_cache.shape[0], generator=mi._gen(84))
    k2 = torch.empty_like(c.k_cache)
    k2[perm] = c.k_cache                      # physical page x moves to perm[x]
    bt2 = perm[c.block_table.long()].to(torch.int32)
    a = ido.dsa_indices_paged(c.q_idx, c.k_cache, c.weights, c.block_table, c.cache_seqlens, 48, c.page)
    b = ido.dsa_indices_paged(c.q_idx, k2, c.weights, bt2, c.cache_seqlens, 48, c.page)
    np.testing.assert_array_equal(a, b)


def pin_paged_unused_slots_never_read():
    """NaN in every slot past a request's length and in the spare pages gives
    the lists of the same cache with finite values there."""
    a = _paged(85, poison=True)
    b = _paged(85, poison=False)
    la = ido.dsa_indices_paged(a.q_idx, a.k_cache, a.weights, a.block_table, a.cache_seqlens, 48, a.page)
    lb = ido.dsa_indices_paged(b.q_idx, b.k_cache, b.weights, b.block_table, b.cache_seqlens, 48, b.page)
    np.testing.assert_array_equal(la, lb)
    assert (la >= 0).sum() > 0


def pin_paged_invalid_pages_never_listed():
    """A page past the block table's width, or a table entry outside the
    pool, gives its positions no key: they are never listed.  Long rows are
    checked against a brute force over the positions that have a key (the
    score written out per head, ranked by score then position), including
    rows with fewer such positions than topk (padded with -1); short rows
    list exactly those positions, in order."""
    c = mi.indexer_paged_case(86, 1, 4, 300, 300, h_idx=8, d_idx=32, topk=40, spare_pages=0, poison=False)
    nb, page, L = c.k_cache.shape[0], c.page, 300
    bt = c.block_table[:, :4].clone()          # positions 256 .. 299 have no page
    bt[0, 1] = -2
    bt[0, 2] = nb + 7
    for topk in (40, 200, 300):
        got = ido.dsa_indices_paged(c.q_idx, c.k_cache, c.weights, bt, c.cache_seqlens, topk, page)
        for j in range(4):
            v = L - 4 + j + 1
            have = [s for s in range(v) if s // page < 4 and 0 <= int(bt[0, s // page]) < nb]
            assert len(have) == 128
            if v <= topk:
                want = have
            else:
                q = c.q_idx[0, j].double().numpy()
                w = c.weights[0, j].double().numpy()
                sc = []
                for s in have:
                    k = c.k_cache[int(bt[0, s // page]), s % page].double().numpy()
                    sc.append((sum(w[h] * max(0.0, float(q[h] @ k)) for h in range(8)), s))
                want = sorted(s for _, s in sorted(sc, key=lambda x: (-x[0], x[1]))[:topk])
            assert got[j].tolist() == want + [-1] * (topk - len(want)), (topk, j)


def pin_selection_never_lists_minus_inf():
    """Hand-worked: -inf positions are not selectable."""
    sc = np.array([3.0, -np.inf, 5.0, -np.inf, 1.0])
    assert ido.select_topk(sc, 2).tolist() == [0, 2]
    assert ido.select_topk(sc, 4).tolist() == [0, 2, 4, -1]
    assert ido.select_topk(np.full(3, -np.inf), 2).tolist() == [-1, -1]
    assert ido.select_topk(np.array([-np.inf, 7.0, 7.0]), 1).tolist() == [1]


def pin_paged_lists_are_never_masked_by_the_forward():
    """The link to the attention's masking: every entry the paged indexer
    lists is a valid entry of the paged forward (the forward oracle's count
    of valid entries equals the number of listed positions), with invalid
    pages in the table, for short and long rows."""
    from oracle import sparse_mla_oracle as orc
    c = mi.indexer_paged_case(87, 3, 4, 100, 400, h_idx=8, d_idx=32, topk=64, spare_pages=1, poison=False)
    nb, page = c.k_cache.shape[0], c.page
    bt = c.block_table[:, :5].clone()
    bt[0, 0] = -1
    bt[1, 3] = nb
    bt[2, 1] = nb + 2
    for topk in (64, 512):
        lst = ido.dsa_indices_paged(c.q_idx, c.k_cache, c.weights, bt, c.cache_seqlens, topk, page)
        idx = torch.from_numpy(lst).reshape(c.q_idx.shape[0], c.q_idx.shape[1], topk).to(torch.int32)
        cnt = orc.valid_count_paged(idx, bt, c.cache_seqlens, page, nb)
        np.testing.assert_array_equal(cnt, (lst >= 0).sum(axis=1))
        assert (lst >= 0).sum() > 0


PINS = [pin_worked_example_scores, pin_worked_example_lists, pin_relu_floor,
        pin_weight_homogeneity_additivity, pin_selection_properties_with_ties,
        pin_selection_matches_torch_topk, pin_visibility_closed_forms,
        pin_scores_selection_consistent, pin_varlen_matches_dense_per_sequence,
        pin_short_rows_reproduce_causal_forward, pin_paged_identity_table_is_dense,
        pin_paged_matches_packed_on_linearised_keys, pin_paged_page_shuffle_invariance,
        pin_paged_unused_slots_never_read, pin_paged_invalid_pages_never_listed,
        pin_selection_never_lists_minus_inf, pin_paged_lists_are_never_masked_by_the_forward]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_indexer_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------

_TS, _SEL, _VIS, _LIN, _PV = (ido.token_scores, ido.select_topk, ido.visible_len, ido.linearise_keys,
                              ido.page_valid)


def _lin_ignores_table(k_cache, block_table, seqlen, page):
    kc = ido._f64(k_cache)
    return np.stack([kc[s // page, s % page] for s in range(seqlen)])


def _lin_table_by_offset(k_cache, block_table, seqlen, page):
    kc = ido._f64(k_cache)
    bt = [int(x) for x in block_table]
    return np.stack([kc[bt[(s % page) % len(bt)], s // page % page] for s in range(seqlen)])


def _ts_no_relu(q_t, w_t, k):
    return (w_t[:, None] * (q_t @ k.T)).sum(axis=0)


def _ts_relu_after_weight(q_t, w_t, k):
    return np.maximum(w_t[:, None] * (q_t @ k.T), 0.0).sum(axis=0)


def _ts_sign(q_t, w_t, k):
    return _TS(-q_t, w_t, k)


def _ts_mean_weight(q_t, w_t, k):
    return _TS(q_t, np.full_like(w_t, w_t.mean()), k)


def _ts_head_transposed(q_t, w_t, k):
    return _TS(q_t, w_t[::-1].copy(), k)


def _sel_ties_to_larger(scores, topk):
    v = scores.shape[0]
    out = np.full(topk, -1, dtype=np.int64)
    order = np.lexsort((-np.arange(v), -scores))
    take = np.sort(order[:min(topk, v)])
    out[:take.shape[0]] = take
    return out


def _sel_smallest(scores, topk):
    return _SEL(-scores, topk)


def _sel_unsorted(scores, topk):
    v = scores.shape[0]
    out = np.full(topk, -1, dtype=np.int64)
    order = np.lexsort((np.arange(v), -scores))[:min(topk, v)]
    out[:order.shape[0]] = order
    return out


def _sel_lists_minus_inf(scores, topk):
    """The previous rule: -inf positions selectable after every other one."""
    v = scores.shape[0]
    out = np.full(topk, -1, dtype=np.int64)
    order = np.lexsort((np.arange(v), -scores))
    take = np.sort(order[:min(topk, v)])
    out[:take.shape[0]] = take
    return out


def _pv_ignores_pool(block_table, seqlen, page, num_blocks):
    return _PV(block_table, seqlen, page, 1 << 30)


def _pv_ignores_width(block_table, seqlen, page, num_blocks):
    bt = [int(x) for x in block_table]
    return np.array([0 <= bt[min(s // page, len(bt) - 1)] < num_blocks for s in range(seqlen)], dtype=bool)


def _short_pad_zero(v, topk):
    out = np.zeros(topk, dtype=np.int64)
    out[:v] = np.arange(v)
    return out


def _short_from_one(v, topk):
    out = np.full(topk, -1, dtype=np.int64)
    out[:v] = np.arange(1, v + 1)
    return out


def _vis_off_by_one(t, s_q, s_kv):
    return int(min(max(t + s_kv - s_q, 0), s_kv))


def _vis_top_left(t, s_q, s_kv):
    return int(min(t + 1, s_kv))


MUTANTS = [("token_scores", _ts_no_relu), ("token_scores", _ts_relu_after_weight),
           ("token_scores", _ts_sign), ("token_scores", _ts_mean_weight),
           ("token_scores", _ts_head_transposed), ("select_topk", _sel_ties_to_larger),
           ("select_topk", _sel_smallest), ("select_topk", _sel_unsorted),
           ("identity_list", _short_pad_zero), ("identity_list", _short_from_one),
           ("linearise_keys", _lin_ignores_table), ("linearise_keys", _lin_table_by_offset),
           ("select_topk", _sel_lists_minus_inf), ("page_valid", _pv_ignores_pool),
           ("page_valid", _pv_ignores_width),
           ("visible_len", _vis_off_by_one),
           ("visible_len", _vis_top_left)]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_indexer_pins_catch_planted_mistake(monkeypatch, name, fn):
    monkeypatch.setattr(ido, name, fn)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, IndexError):     # a pin the mistake breaks, or one it crashes
            failed += 1
    assert failed >= 1, f"no pin caught the planted mistake {fn.__name__}"
