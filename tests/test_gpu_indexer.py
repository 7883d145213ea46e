"""GPU parity of the DSA indexer (dsa_indexer_scores, dsa_topk,
dsa_indexer_topk through the C ABI) against the float64 oracle on the same
seeded inputs.

* Selection alone is integer work: on fp32 scores given to both sides (tied
  integer levels, -inf holes, distinct normal draws, rows past the
  shared-memory staging size) the lists must be identical.
* Scores: per element, |gpu - oracle| <= sum_j |w_j| (2^-16 sum_d |q_jd k_d|)
  + 2^-18 sum_j |w_j| relu(q_j . k): the worst case of an fp32 sum of 128
  bf16 products (each exact in fp32) in any order even with truncating
  adders (128 * 2^-23), then the fp32 weighted sum of H_I terms.
* Lists from GPU scores: valid lists (increasing, distinct, visible, the
  right count; short rows the identity list), every selected position's
  oracle score at least every unselected one's up to the two bounds, and
  identical to the oracle's list wherever the oracle's gap at the top-k
  boundary exceeds twice the row's largest bound.
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi
from oracle import dsa_indexer_oracle as ido

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GAMMA_DOT = 2.0 ** -16
GAMMA_SUM = 2.0 ** -18


@pytest.fixture(scope="module")
def smla(cuda_lib):
    import serving_sparse_mla_gb300 as pkg
    pkg.clear_device_error()
    yield pkg
    assert pkg.get_device_error() == 0


def _dev(c):
    cq = None if c.cu_seqlens_q is None else c.cu_seqlens_q.to(DEV)
    ck = None if c.cu_seqlens_kv is None else c.cu_seqlens_kv.to(DEV)
    return c.q_idx.to(DEV), c.k_idx.to(DEV), c.weights.to(DEV), cq, ck


def _row_meta(c, r):
    """(sequence KV start, visible length) of packed row r."""
    if c.cu_seqlens_q is None:
        return 0, ido.visible_len(r, c.q_idx.shape[0], c.k_idx.shape[0])
    cq, ck = c.cu_seqlens_q.tolist(), c.cu_seqlens_kv.tolist()
    b = int(np.searchsorted(cq, r, side="right")) - 1
    return ck[b], ido.visible_len(r - cq[b], cq[b + 1] - cq[b], ck[b + 1] - ck[b])


def _row_ref(c, r):
    """Oracle scores of row r over its visible positions and their bounds."""
    k0, v = _row_meta(c, r)
    q = c.q_idx[r].double().numpy()
    w = c.weights[r].double().numpy()
    k = c.k_idx[k0:k0 + v].double().numpy()
    ref = ido.token_scores(q, w, k)
    dots = q @ k.T
    bound = np.abs(w) @ (GAMMA_DOT * (np.abs(q) @ np.abs(k).T)) + GAMMA_SUM * (np.abs(w) @ np.maximum(dots, 0.0))
    return ref, bound + 1e-30, v


def _check_scores(c, got, rows, row0=0):
    for r in rows:
        ref, bound, v = _row_ref(c, r)
        g = got[r - row0]
        err = np.abs(g[:v].astype(np.float64) - ref)
        bad = np.nonzero(err > bound)[0]
        assert bad.size == 0, (f"row {r}: {bad.size} scores off, first pos {bad[0]}: gpu {g[bad[0]]} "
                               f"oracle {ref[bad[0]]} bound {bound[bad[0]]}")
        assert np.all(np.isneginf(g[v:])), f"row {r}: positions past {v} were written"


def _check_list(c, lst, r, topk):
    """Validity, ordering against the oracle scores, exactness when unique.
    Returns True when the row was checked exactly."""
    _, v = _row_meta(c, r)
    lst = np.asarray(lst)
    n = min(topk, v)
    assert np.all(lst[n:] == -1), f"row {r}: padding"
    sel = lst[:n]
    assert np.all(sel >= 0) and np.all(sel < v), f"row {r}: out of range"
    assert np.all(np.diff(sel) > 0), f"row {r}: not increasing"
    if v <= topk:
        np.testing.assert_array_equal(sel, np.arange(v))
        return True
    ref, bound, _ = _row_ref(c, r)
    chosen = np.zeros(v, dtype=bool)
    chosen[sel] = True
    lo = (ref + bound)[chosen].min()
    hi = (ref - bound)[~chosen].max()
    assert lo >= hi, f"row {r}: a selected score falls below an unselected one beyond the bounds"
    srt = np.sort(ref)[::-1]
    if srt[topk - 1] - srt[topk] > 2.0 * bound.max():
        np.testing.assert_array_equal(sel, ido.select_topk(ref, topk)[:n])
        return True
    return False


# --------------------------------------------------------------------------- selection alone

def _lens_dense(s_q, s_kv):
    return [ido.visible_len(t, s_q, s_kv) for t in range(s_q)]


@pytest.mark.parametrize("rows,width,topk", [(40, 300, 16), (64, 3000, 2048), (33, 2500, 1),
                                             (20, 2049, 2048), (24, 700, 650)])
def test_topk_tied_scores_exact(smla, rows, width, topk):
    """Integer levels with many ties at the threshold and -inf holes."""
    sc = mi.tied_scores(rows * 7 + width, rows, width)
    got = smla.dsa_topk(sc.to(DEV), topk, rows, width).cpu().numpy()
    ref = ido.topk_rows(sc.numpy(), _lens_dense(rows, width), topk)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("rows,width", [(12, 20000), (4, 60000)])
def test_topk_long_rows_exact(smla, rows, width):
    """Distinct normal scores on rows past 8192 positions (1024-thread CTAs):
    staged in shared memory up to 49152 positions, read from global memory
    on every pass beyond."""
    g = torch.Generator().manual_seed(501 + width)
    topk = 2048
    sc = torch.randn((rows, width), generator=g)
    got = smla.dsa_topk(sc.to(DEV), topk, rows, width).cpu().numpy()
    ref = ido.topk_rows(sc.numpy(), _lens_dense(rows, width), topk)
    np.testing.assert_array_equal(got, ref)


def test_topk_constant_row_takes_first_positions(smla):
    """A constant row takes its first positions; a row of -inf selects
    nothing (-inf is never selectable); a row with fewer finite scores than
    topk lists those and pads with -1."""
    sc = torch.zeros((4, 5000))
    sc[1] = float("-inf")
    sc[3] = float("-inf")
    sc[3, 4000:4030] = 1.0
    got = smla.dsa_topk(sc.to(DEV), 100, 4, 5000).cpu().numpy()
    for i in (0, 2):
        np.testing.assert_array_equal(got[i], np.arange(100))
    assert np.all(got[1] == -1)
    np.testing.assert_array_equal(got[3], np.concatenate([np.arange(4000, 4030), np.full(70, -1)]))


def test_topk_varlen_exact(smla):
    q_lens, kv_lens = [3, 40, 1, 17, 60], [3, 900, 2100, 40, 60]
    cq = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    ck = torch.tensor(np.concatenate([[0], np.cumsum(kv_lens)]), dtype=torch.int32)
    total_q, total_kv, width = int(cq[-1]), int(ck[-1]), max(kv_lens)
    sc = mi.tied_scores(502, total_q, width, levels=40)
    lens = []
    for b in range(5):
        lens += [ido.visible_len(t, q_lens[b], kv_lens[b]) for t in range(q_lens[b])]
    got = smla.dsa_topk(sc.to(DEV), 32, total_q, total_kv, cq.to(DEV), ck.to(DEV)).cpu().numpy()
    np.testing.assert_array_equal(got, ido.topk_rows(sc.numpy(), lens, 32))


def test_topk_row_range(smla):
    """Only rows row0 .. row0 + n_rows - 1 are written."""
    sc = mi.tied_scores(503, 10, 400)
    out = torch.full((30, 64), -7, dtype=torch.int32, device=DEV)
    smla.dsa_topk(sc.to(DEV), 64, 30, 400, row0=12, n_rows=10, indices=out)
    o = out.cpu().numpy()
    assert np.all(o[:12] == -7) and np.all(o[22:] == -7)
    lens = [ido.visible_len(t, 30, 400) for t in range(12, 22)]
    np.testing.assert_array_equal(o[12:22], ido.topk_rows(sc.numpy(), lens, 64))


# --------------------------------------------------------------------------- scores

@pytest.mark.parametrize("h_idx", [64, 32, 16])
def test_scores_dense(smla, h_idx):
    """Several 128-position tiles and chunks of 2048, ragged tails, a cached
    prefix (s_kv > s_q), every row scored."""
    c = mi.indexer_case(510 + h_idx, 37, 2300, h_idx=h_idx)
    got = smla.dsa_indexer_scores(*_dev(c)).cpu().numpy()
    _check_scores(c, got, range(37))


def test_scores_square_causal_and_empty_rows(smla):
    c = mi.indexer_case(520, 300, 260)    # 40 queries before position 0 see nothing
    got = smla.dsa_indexer_scores(*_dev(c)).cpu().numpy()
    _check_scores(c, got, list(range(0, 45)) + list(range(290, 300)))


def test_scores_skip_len_and_row_range(smla):
    c = mi.indexer_case(521, 200, 200)
    got = smla.dsa_indexer_scores(*_dev(c), row0=50, n_rows=101, skip_len=100).cpu().numpy()
    assert got.shape[0] == 101
    assert np.all(np.isneginf(got[:50]))           # rows 50..99 see <= 100 positions: skipped
    _check_scores(c, got, range(100, 151), row0=50)


def test_scores_varlen_groups_straddle_sequences(smla):
    c = mi.indexer_varlen_case(522, [5, 130, 3, 77, 1], [300, 130, 2100, 77, 9])
    got = smla.dsa_indexer_scores(*_dev(c)).cpu().numpy()
    _check_scores(c, got, range(int(c.cu_seqlens_q[-1])))


# --------------------------------------------------------------------------- lists

def test_indexer_topk_dense(smla):
    c = mi.indexer_case(530, 600, 2600, topk=2048)     # rows 0..47 short, the rest scored
    lst = smla.dsa_indexer_topk(*_dev(c)[:3], 2048).cpu().numpy()
    exact = sum(_check_list(c, lst[r], r, 2048) for r in range(0, 600, 7))
    assert exact >= 25


def test_indexer_topk_chunked_equals_unchunked(smla):
    c = mi.indexer_case(531, 300, 2400, topk=512)
    q, k, w, _, _ = _dev(c)
    full = smla.dsa_indexer_topk(q, k, w, 512)
    ws = torch.empty(7 * 2400 * 4 + 5, dtype=torch.uint8, device=DEV)    # 7 rows of logits per chunk
    part = smla.dsa_indexer_topk(q, k, w, 512, workspace=ws)
    assert torch.equal(full, part)
    for r in (0, 1, 150, 299):
        _check_list(c, full[r].cpu().numpy(), r, 512)


def test_indexer_topk_varlen(smla):
    c = mi.indexer_varlen_case(532, [50, 300, 9, 200], [3000, 300, 2500, 200], topk=256)
    q, k, w, cq, ck = _dev(c)
    lst = smla.dsa_indexer_topk(q, k, w, 256, cq, ck).cpu().numpy()
    exact = sum(_check_list(c, lst[r], r, 256) for r in range(0, 559, 3))
    assert exact >= 120


def test_indexer_topk_all_short(smla):
    """Every row sees <= topk positions: identity lists, no workspace."""
    c = mi.indexer_case(533, 100, 120, topk=2048)
    lst = smla.dsa_indexer_topk(*_dev(c)[:3], 2048, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    lst = lst.cpu().numpy()
    for r in range(100):
        v = ido.visible_len(r, 100, 120)
        np.testing.assert_array_equal(lst[r, :v], np.arange(v))
        assert np.all(lst[r, v:] == -1)


def test_indexer_topk_full_size_sampled(smla):
    """The 8192-token prefill at topk 2048 with 64 indexer heads, in 1024-row
    logits chunks; sampled rows against the oracle."""
    c = mi.indexer_case(534, 8192, 8192, topk=2048)
    q, k, w, _, _ = _dev(c)
    ws = torch.empty(1024 * 8192 * 4, dtype=torch.uint8, device=DEV)
    lst = smla.dsa_indexer_topk(q, k, w, 2048, workspace=ws).cpu().numpy()
    rows = [0, 2047, 2048, 2049, 3000, 4095, 5555, 8191]
    exact = sum(_check_list(c, lst[r], r, 2048) for r in rows)
    assert exact >= 3


# --------------------------------------------------------------------------- edge cases

def test_indexer_varlen_edge_sequences(smla):
    """Empty query runs, empty key runs, fewer keys than queries (the first
    queries see nothing), single-token sequences, 16 indexer heads."""
    q_lens = [0, 7, 3, 0, 40, 1, 9]
    kv_lens = [5, 0, 2, 0, 700, 1, 300]
    c = mi.indexer_varlen_case(540, q_lens, kv_lens, h_idx=16, topk=64)
    q, k, w, cq, ck = _dev(c)
    lst = smla.dsa_indexer_topk(q, k, w, 64, cq, ck).cpu().numpy()
    for r in range(int(c.cu_seqlens_q[-1])):
        _check_list(c, lst[r], r, 64)
    got = smla.dsa_indexer_scores(q, k, w, cq, ck).cpu().numpy()
    _check_scores(c, got, range(int(c.cu_seqlens_q[-1])))


def test_indexer_many_short_sequences(smla):
    """Hundreds of short sequences: most groups straddle several."""
    g = torch.Generator().manual_seed(541)
    q_lens = torch.randint(1, 12, (300,), generator=g).tolist()
    kv_lens = [ql + int(x) for ql, x in zip(q_lens, torch.randint(0, 90, (300,), generator=g).tolist())]
    c = mi.indexer_varlen_case(541, q_lens, kv_lens, h_idx=32, topk=40)
    q, k, w, cq, ck = _dev(c)
    lst = smla.dsa_indexer_topk(q, k, w, 40, cq, ck).cpu().numpy()
    total = int(c.cu_seqlens_q[-1])
    exact = sum(_check_list(c, lst[r], r, 40) for r in range(0, total, 5))
    assert exact >= total // 5 // 2


def test_indexer_varlen_chunked_and_long_stride(smla):
    """A logits budget of a few rows, and a row length above the longest
    sequence, give the lists of the one-chunk call."""
    c = mi.indexer_varlen_case(542, [30, 200, 17], [2500, 200, 3100], topk=256)
    q, k, w, cq, ck = _dev(c)
    full = smla.dsa_indexer_topk(q, k, w, 256, cq, ck)
    ws = torch.empty(5 * 3104 * 4, dtype=torch.uint8, device=DEV)
    part = smla.dsa_indexer_topk(q, k, w, 256, cq, ck, workspace=ws)
    wide = smla.dsa_indexer_topk(q, k, w, 256, cq, ck, max_seqlen_kv=3500)
    assert torch.equal(full, part) and torch.equal(full, wide)
    for r in (0, 29, 30, 100, 229, 230, 246):
        _check_list(c, full[r].cpu().numpy(), r, 256)


def test_indexer_row_length_too_small_is_reported(smla):
    """A max_seqlen_kv below the longest sequence cuts rows to it (nothing is
    written past a logits row) and records the error code 0x611."""
    c = mi.indexer_varlen_case(543, [20, 20], [600, 3000], topk=128)
    q, k, w, cq, ck = _dev(c)
    smla.clear_device_error()
    lst = smla.dsa_indexer_topk(q, k, w, 128, cq, ck, max_seqlen_kv=1000)
    torch.cuda.synchronize()
    assert smla.get_device_error() == 0x611
    smla.clear_device_error()
    lst = lst.cpu().numpy()
    for r in range(20):             # the first sequence fits: exact rules
        _check_list(c, lst[r], r, 128)
    assert np.all((lst[20:] >= 0) & (lst[20:] < 1000))   # cut rows still list valid positions


def test_indexer_lists_drive_the_forward(smla):
    """The pipeline: GPU lists into the sparse forward equal the oracle's
    forward over the oracle's lists on every row whose list is unique."""
    from oracle import sparse_mla_oracle as orc
    s, topk = 300, 128
    c = mi.indexer_case(544, s, s, topk=topk)
    lst = smla.dsa_indexer_topk(*_dev(c)[:3], topk)
    ref_lst = ido.dsa_indices(c.q_idx, c.k_idx, c.weights, topk)
    same = [r for r in range(s) if np.array_equal(lst[r].cpu().numpy(), ref_lst[r])]
    assert len(same) >= s // 2
    g = mi._gen(545)
    q = mi.randn_bf16(g, (s, 8, mi.D_QK))
    kv = mi.randn_bf16(g, (s, mi.D_QK))
    out, lse = smla.sparse_mla_fwd(q.to(DEV), kv.to(DEV), lst, mi.default_sm_scale())
    ro, rl = orc.sparse_mla_fwd(q, kv, torch.from_numpy(ref_lst).to(torch.int32), mi.default_sm_scale(),
                                tokens=same)
    o = out.float().cpu().numpy()[same]
    l = lse.cpu().numpy()[same]
    assert np.all(np.abs(o - ro) <= 2e-2 + 2e-2 * np.abs(ro))
    assert np.all(np.abs(l - rl) <= 1e-3)


# --------------------------------------------------------------------------- paged (decode) cache

def _pdev(c):
    return (c.q_idx.to(DEV), c.k_cache.to(DEV), c.weights.to(DEV), c.block_table.to(DEV), c.cache_seqlens.to(DEV))


def _paged_row_ref(c, r, keys_cache, block_table=None):
    """Oracle scores of decode row r (-inf where a position has no key),
    their per-element bounds and the row's visible length."""
    bt = c.block_table if block_table is None else block_table
    s_next = c.q_idx.shape[1]
    b, j = divmod(r, s_next)
    lk = int(c.cache_seqlens[b])
    v = ido.visible_len(j, s_next, lk)
    if b not in keys_cache:
        keys_cache[b] = ido.linearise_keys(c.k_cache, bt[b], lk, c.page)
    k = keys_cache[b][:v]
    q = c.q_idx[b, j].double().numpy()
    w = c.weights[b, j].double().numpy()
    ref = ido.paged_row_scores(q, w, k, ido.page_valid(bt[b], v, c.page, c.k_cache.shape[0]))
    bound = np.abs(w) @ (GAMMA_DOT * (np.abs(q) @ np.abs(k).T)) + GAMMA_SUM * (np.abs(w) @ np.maximum(q @ k.T, 0.0))
    return ref, bound + 1e-30, v


def _check_paged_list(c, lst, r, topk, keys_cache, block_table=None):
    """Validity of one decode row's list (only positions with a key, in
    order, -1 padded), its order within the score bounds, and equality with
    the oracle's list where the oracle's top-k boundary gap exceeds twice the
    bound.  Returns whether the row was compared exactly."""
    ref, bound, v = _paged_row_ref(c, r, keys_cache, block_table)
    lst = np.asarray(lst)
    keyed = np.nonzero(~np.isneginf(ref))[0]
    n = min(topk, keyed.size)
    assert np.all(lst[n:] == -1), f"row {r}: padding"
    sel = lst[:n]
    assert np.all(np.isin(sel, keyed)) and np.all(np.diff(sel) > 0), f"row {r}: invalid list"
    if keyed.size <= topk:
        np.testing.assert_array_equal(sel, keyed)
        return True
    chosen = np.zeros(v, dtype=bool)
    chosen[sel] = True
    others = ~chosen & ~np.isneginf(ref)
    assert (ref + bound)[chosen].min() >= (ref - bound)[others].max(), f"row {r}: order beyond the bounds"
    srt = np.sort(ref[keyed])[::-1]
    if srt[topk - 1] - srt[topk] > 2.0 * bound.max():
        np.testing.assert_array_equal(sel, ido.select_topk(ref, topk)[:n])
        return True
    return False


def test_paged_scores(smla):
    """Every row scored over its pages (NaN in every unused slot and spare
    page), positions past a row's length untouched."""
    c = mi.indexer_paged_case(550, 5, 6, 300, 1500, topk=128)
    max_len = int(c.cache_seqlens.max())
    got = smla.dsa_indexer_scores_paged(*_pdev(c), max_len).cpu().numpy()
    keys = {}
    for r in range(30):
        ref, bound, v = _paged_row_ref(c, r, keys)
        assert not np.isneginf(ref).any()
        err = np.abs(got[r, :v].astype(np.float64) - ref)
        assert np.all(err <= bound), f"row {r}: max err {err.max()}"
        assert np.all(np.isneginf(got[r, v:]))


def test_paged_invalid_pages_score_minus_inf_and_are_never_listed(smla):
    """A block table with entries -1 and num_blocks + 3 and a width below the
    requests' lengths: the positions of those pages score exactly -inf, every
    other visible position within the bound; the lists hold only keyed
    positions (exactly the oracle's list where it is unique), and every
    listed entry is one the paged forward counts as valid (the forward's
    valid-count export equals the number of listed entries)."""
    c = mi.indexer_paged_case(556, 4, 6, 300, 1600, topk=256)
    nb = c.k_cache.shape[0]
    W = 12                                            # positions >= 768 have no page
    bt = c.block_table[:, :W].clone()
    bt[0, 2] = -1
    bt[1, 0] = nb + 3
    bt[2, 5] = -1
    bt[3, 1] = nb
    max_len = int(c.cache_seqlens.max())
    d = lambda t: t.to(DEV)
    q, k, w, _, sl = _pdev(c)
    got = smla.dsa_indexer_scores_paged(q, k, w, d(bt), sl, max_len).cpu().numpy()
    keys = {}
    for r in range(24):
        ref, bound, v = _paged_row_ref(c, r, keys, bt)
        none = np.isneginf(ref)
        assert np.all(np.isneginf(got[r, :v][none])), f"row {r}: a position without a key scored"
        err = np.abs(got[r, :v][~none].astype(np.float64) - ref[~none])
        assert np.all(err <= bound[~none]), f"row {r}: max err {err.max()}"
    for topk in (256, 2048):   # long rows, and rows with fewer keyed positions than topk
        lst = smla.dsa_indexer_topk_paged(q, k, w, d(bt), sl, topk).cpu()
        keys = {}
        for r in range(24):
            _check_paged_list(c, lst.reshape(24, topk)[r].numpy(), r, topk, keys, bt)
        idx = lst.reshape(4, 6, topk).to(DEV)
        counts = smla.debug_valid_count_paged(idx, d(bt), sl, c.page, nb).cpu().numpy()
        np.testing.assert_array_equal(counts, (lst.reshape(24, topk).numpy() >= 0).sum(axis=1))


def test_paged_lists_and_page_shuffle(smla):
    c = mi.indexer_paged_case(551, 7, 6, 700, 3000, topk=512)
    q, k, w, bt, sl = _pdev(c)
    lst = smla.dsa_indexer_topk_paged(q, k, w, bt, sl, 512).cpu().numpy().reshape(42, 512)
    keys = {}
    exact = sum(_check_paged_list(c, lst[r], r, 512, keys) for r in range(42))
    assert exact >= 6   # the oracle's gaps make 8 of these rows unique
    # a shuffle of the physical pages, the block table remapped: same lists
    perm = torch.randperm(c.k_cache.shape[0], generator=mi._gen(552))
    k2 = torch.empty_like(c.k_cache)
    k2[perm] = c.k_cache
    bt2 = perm[c.block_table.long()].to(torch.int32)
    lst2 = smla.dsa_indexer_topk_paged(q, k2.to(DEV), w, bt2.to(DEV), sl, 512).cpu().numpy().reshape(42, 512)
    np.testing.assert_array_equal(lst, lst2)


def test_paged_short_requests_and_budget(smla):
    """Requests shorter than topk (identity lists), one shorter than its MTP
    rows (its first rows see nothing), and a logits budget of three rows."""
    c = mi.indexer_paged_case(553, 4, 6, 3, 900, topk=256)
    c.cache_seqlens[1] = 4          # rows 0, 1 of request 1 see no position
    c.cache_seqlens[2] = 200        # short: identity lists
    q, k, w, bt, sl = _pdev(c)
    full = smla.dsa_indexer_topk_paged(q, k, w, bt, sl, 256)
    ws = torch.empty(3 * 904 * 4, dtype=torch.uint8, device=DEV)
    part = smla.dsa_indexer_topk_paged(q, k, w, bt, sl, 256, max_seqlen_kv=900, workspace=ws)
    assert torch.equal(full, part)
    lst = full.cpu().numpy().reshape(24, 256)
    keys = {}
    for r in range(24):
        _check_paged_list(c, lst[r], r, 256, keys)
    assert np.all(lst[6:8] == -1)


def test_paged_decode_shape_sampled(smla):
    """16 requests x 6 MTP tokens, contexts U[4096, 32768], topk 2048, 64
    indexer heads (the decode workload's shape); sampled rows."""
    c = mi.indexer_paged_case(554, 16, 6, 4096, 32768, topk=2048)
    lst = smla.dsa_indexer_topk_paged(*_pdev(c), 2048).cpu().numpy().reshape(96, 2048)
    keys = {}
    # rows of ~4-33 K positions: the oracle's gap at the 2048th score is
    # within the bounds, so each row is checked by its validity and ordering
    for r in (0, 5, 17, 40, 63, 95):
        _check_paged_list(c, lst[r], r, 2048, keys)
