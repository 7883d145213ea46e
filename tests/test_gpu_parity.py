"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs (tolerances in tests/parity.py)."""
import math

import numpy as np
import pytest
import torch

import mla_inputs as mi
from oracle import sparse_mla_oracle as orc
from tests.oracle_pool import check_all_tokens
from tests.parity import compare, pv_rounding_sigma, record, tight_ratio

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run_fwd(smla, case, kv=None, indices=None):
    kv = case.kv if kv is None else kv
    idx = case.indices if indices is None else indices
    out, lse = smla.sparse_mla_fwd(case.q.to(DEV), kv.to(DEV), idx.to(DEV), case.sm_scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _check_fwd(smla, case, kv=None, indices=None, tokens=None, what=""):
    kv = case.kv if kv is None else kv
    idx = case.indices if indices is None else indices
    o, l = _run_fwd(smla, case, kv, idx)
    if tokens is not None:
        o, l = o[tokens], l[tokens]
    ref_o, ref_l = orc.sparse_mla_fwd(case.q, kv, idx, case.sm_scale, tokens=tokens)
    return compare(o, l, ref_o, ref_l, what or case.name)


@pytest.fixture(scope="module")
def smla(cuda_lib):
    import serving_sparse_mla_gb300 as pkg
    pkg.clear_device_error()
    yield pkg
    assert pkg.get_device_error() == 0


# ---------------------------------------------------------------- dense prefill

def test_tiny_prefill_config(smla):
    """s_q = s_kv = 64, h = 8, topk = 2048: every causal position listed."""
    _check_fwd(smla, mi.config(1))


@pytest.mark.parametrize("h_q", [1, 8, 16, 24, 64, 100, 128])
def test_head_counts(smla, h_q):
    case = mi.prefill_case(200 + h_q, s_q=37, s_kv=420, h_q=h_q, topk=384)
    _check_fwd(smla, case)


@pytest.mark.parametrize("topk", [1, 64, 128, 192, 300, 2048])
def test_topk_values(smla, topk):
    case = mi.prefill_case(300 + topk, s_q=160, s_kv=700, h_q=8, topk=topk)
    _check_fwd(smla, case)


def test_scattered_padding_and_poisoned_rows(smla):
    """-1 anywhere in the list; every KV row no list references is NaN."""
    case = mi.prefill_case(401, s_q=200, s_kv=900, h_q=8, topk=512)
    idx = mi.scatter_padding(mi._gen(402), case.indices)
    kv = mi.poison_unreferenced(case.kv, case.referenced)
    _check_fwd(smla, case, kv=kv, indices=idx)


def test_masking_edge_cases(smla):
    s_q, s_kv, topk = 8, 50, 256
    case = mi.prefill_case(403, s_q=s_q, s_kv=s_kv, h_q=16, topk=topk)
    idx = torch.full((s_q, topk), -1, dtype=torch.int32)
    idx[1, 200] = 7                                   # single valid entry, late block
    idx[2, :] = torch.randint(-9, -1, (topk,), dtype=torch.int32)    # all negative
    idx[3, :] = torch.randint(s_kv, s_kv + 1000, (topk,), dtype=torch.int32)  # all past the end
    idx[4, :5] = torch.tensor([3, 3, 3, 9, 9])       # duplicates
    idx[5, 0::2] = torch.arange(0, topk // 2, dtype=torch.int32) % s_kv   # every other entry
    idx[6, :] = torch.arange(topk, dtype=torch.int32) % s_kv            # all valid, repeats
    idx[7, 127:129] = torch.tensor([11, 12])          # straddles a 128-entry block edge
    kv = mi.poison_unreferenced(case.kv, torch.unique(idx[(idx >= 0) & (idx < s_kv)]))
    o, l = _run_fwd(smla, case, kv, idx)
    ref_o, ref_l = orc.sparse_mla_fwd(case.q, kv, idx, case.sm_scale)
    compare(o, l, ref_o, ref_l, "masking")
    # rows 0, 2, 3: nothing valid -> exactly +0 and -inf
    for t in (0, 2, 3):
        assert np.all(o[t] == 0.0) and np.all(np.isneginf(l[t]))
    # row 1: a single valid entry returns that value row (bf16-exact)
    assert np.array_equal(o[1], np.broadcast_to(case.kv[7, :512].float().numpy(), o[1].shape))


def test_long_lists_span_several_windows(smla):
    """top-k lists longer than 32 blocks of 64 (the producer scans them 32
    blocks at a time), a ragged last block, and lists whose only valid
    entries sit late: in the second window, or in one block after -1s."""
    s_q, s_kv, topk = 24, 6000, 3100
    case = mi.prefill_case(404, s_q=s_q, s_kv=s_kv, h_q=8, topk=topk)
    idx = case.indices.clone()
    g = torch.Generator().manual_seed(405)
    idx[0, :] = -1
    idx[0, 3000:3003] = torch.tensor([5, 4000, 5999], dtype=torch.int32)   # second window, ragged block
    idx[1, :2500] = -1                                                        # first window empty
    idx[1, 2500:] = torch.randint(0, s_kv, (topk - 2500,), generator=g, dtype=torch.int32)
    idx[2, :] = -1
    idx[2, 1500:1564] = torch.randint(0, s_kv, (64,), generator=g, dtype=torch.int32)  # one block, mid window
    idx[3, :] = torch.randint(0, s_kv, (topk,), generator=g, dtype=torch.int32)        # every block valid
    idx[3, 64:2048] = -1
    kv = mi.poison_unreferenced(case.kv, torch.unique(idx[(idx >= 0) & (idx < s_kv)]))
    o, l = _run_fwd(smla, case, kv, idx)
    ref_o, ref_l = orc.sparse_mla_fwd(case.q, kv, idx, case.sm_scale)
    compare(o, l, ref_o, ref_l, "long lists")


def test_s_kv_zero_and_empty_batch(smla):
    q = torch.randn(3, 8, 576, device=DEV).to(torch.bfloat16)
    kv = torch.empty(0, 576, device=DEV, dtype=torch.bfloat16)
    idx = torch.zeros(3, 64, dtype=torch.int32, device=DEV)
    out, lse = smla.sparse_mla_fwd(q, kv, idx, 0.1)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    out, lse = smla.sparse_mla_fwd(q[:0], kv, idx[:0], 0.1)
    assert out.shape == (0, 8, 512)


def _check_whole(name, layout, q, kv, indices, out, lse, sm_scale, extra=None):
    """Every token of a full-size workload against the oracle on the host
    cores: the allclose bar on every element, and the tight check of
    tests/parity.py (its worst ratio recorded, and required <= 1)."""
    st = check_all_tokens(layout, q, kv, indices, out.cpu(), lse.cpu(), sm_scale, extra)
    assert st["fail"] is None, st["fail"]
    assert st["tokens"] == q.shape[0]
    record(name, tokens=st["tokens"], max_dout=st["max_dout"], max_dlse=st["max_dlse"],
           tight_ratio=st["tight"], tight_ratio_full_lists=st["tight_full"])
    assert st["tight"] <= 1.0, f"{name}: tight check ratio {st['tight']:.3f}"
    return st


def test_tiny_prefill_config_tight(smla):
    case = mi.config(1)
    out, lse = smla.sparse_mla_fwd(case.q.to(DEV), case.kv.to(DEV), case.indices.to(DEV), case.sm_scale)
    _check_whole("config 1 tiny prefill", "dense", case.q, case.kv, case.indices, out, lse, case.sm_scale)


def test_mid_prefill_config_all_tokens(smla):
    """s_q = s_kv = 2119, h = 8, topk = 2048 (the pages' SWE-like shape):
    every token, with the tight check (72 tokens list 2048 valid entries)."""
    case = mi.config(2)
    out, lse = smla.sparse_mla_fwd(case.q.to(DEV), case.kv.to(DEV), case.indices.to(DEV), case.sm_scale)
    st = _check_whole("config 2 mid prefill", "dense", case.q, case.kv, case.indices, out, lse, case.sm_scale)
    assert st["tight_full"] > 0.0   # the full-list tokens were checked


def test_wide_head_config_all_tokens(smla):
    """s_q = s_kv = 8192, h = 64, topk = 2048 at the launch the bench times:
    every token against the oracle (host cores), with the tight check."""
    case = mi.config(3)
    out, lse = smla.sparse_mla_fwd(case.q.to(DEV), case.kv.to(DEV), case.indices.to(DEV), case.sm_scale)
    _check_whole("config 3 wide-head prefill", "dense", case.q, case.kv, case.indices, out, lse, case.sm_scale)


# ---------------------------------------------------------------- indices-free causal mode

@pytest.mark.parametrize("s_q,s_kv,h_q", [(64, 64, 8), (300, 300, 8), (100, 700, 64), (37, 20, 16), (1, 2500, 8)])
def test_causal_mode(smla, s_q, s_kv, h_q):
    """Every query attends to all KV positions at or before its own (queries
    are the last s_q positions; with s_q > s_kv the first ones see nothing);
    one query over 2500 positions spans two scan windows."""
    case = mi.prefill_case(800 + s_q, s_q=s_q, s_kv=s_kv, h_q=h_q, topk=64)
    out, lse = smla.sparse_mla_fwd_causal(case.q.to(DEV), case.kv.to(DEV), case.sm_scale)
    torch.cuda.synchronize()
    ref_o, ref_l = orc.causal_mla_fwd(case.q, case.kv, case.sm_scale)
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, f"causal {s_q}x{s_kv}")


def test_causal_mode_equals_sparse_with_full_causal_lists(smla):
    """The causal mode walks the same blocks as the sparse forward given each
    token's causal positions in order, so the two agree bit for bit."""
    s = 300
    case = mi.prefill_case(810, s_q=s, s_kv=s, h_q=8, topk=64)
    idx = torch.full((s, s), -1, dtype=torch.int32)
    for t in range(s):
        idx[t, : t + 1] = torch.arange(t + 1, dtype=torch.int32)
    q, kv = case.q.to(DEV), case.kv.to(DEV)
    o1, l1 = smla.sparse_mla_fwd_causal(q, kv, case.sm_scale)
    o2, l2 = smla.sparse_mla_fwd(q, kv, idx.to(DEV), case.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ---------------------------------------------------------------- packed prefill

def _check_varlen(smla, case, tokens=None, what=""):
    d = lambda t: t.to(DEV)
    out, lse = smla.sparse_mla_fwd_varlen(d(case.q), d(case.kv), d(case.indices), d(case.cu_seqlens_q),
                                          d(case.cu_seqlens_kv), case.sm_scale)
    torch.cuda.synchronize()
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    if tokens is not None:
        o, l = o[tokens], l[tokens]
    ref_o, ref_l = orc.sparse_mla_fwd_varlen(case.q, case.kv, case.indices, case.cu_seqlens_q,
                                             case.cu_seqlens_kv, case.sm_scale, tokens=tokens)
    return compare(o, l, ref_o, ref_l, what or case.name)


@pytest.mark.parametrize("h_q", [8, 64])
def test_varlen_small(smla, h_q):
    case = mi.varlen_case(500 + h_q, [130, 1, 257, 64, 300], h_q, topk=256)
    case.kv = mi.poison_unreferenced(case.kv, case.referenced)
    _check_varlen(smla, case)


def test_varlen_chunked_lengths_and_empty_sequences(smla):
    """Packed prefill with query and KV lengths that differ per sequence (a
    chunk of queries over a longer KV history), a sequence with neither, one
    with KV rows but no queries, and one with queries but no KV rows (every
    entry masked: out 0, LSE -inf).  Lists hold distinct in-range local
    positions, some past the sequence's KV end (masked), and -1 padding."""
    lens_q = [100, 0, 0, 37, 10, 5]
    lens_kv = [300, 0, 50, 0, 64, 700]
    topk = 256
    g = torch.Generator().manual_seed(640)
    total_q, total_kv = sum(lens_q), sum(lens_kv)
    q = torch.randn((total_q, 8, 576), generator=g).to(torch.bfloat16)
    kv = torch.randn((total_kv, 576), generator=g).to(torch.bfloat16)
    idx = torch.full((total_q, topk), -1, dtype=torch.int32)
    t = 0
    for lq, lk in zip(lens_q, lens_kv):
        for _ in range(lq):
            n = min(topk - 8, lk)
            if n:
                idx[t, :n] = torch.randperm(lk, generator=g)[:n].to(torch.int32)
            idx[t, n:n + 8] = lk + torch.arange(8, dtype=torch.int32)   # past this sequence's KV end
            t += 1
    cu_q = torch.tensor([0] + np.cumsum(lens_q).tolist(), dtype=torch.int32)
    cu_kv = torch.tensor([0] + np.cumsum(lens_kv).tolist(), dtype=torch.int32)
    sm_scale = 1.0 / math.sqrt(576)
    d = lambda x: x.to(DEV)
    out, lse = smla.sparse_mla_fwd_varlen(d(q), d(kv), d(idx), d(cu_q), d(cu_kv), sm_scale)
    torch.cuda.synchronize()
    ref_o, ref_l = orc.sparse_mla_fwd_varlen(q, kv, idx, cu_q, cu_kv, sm_scale)
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "varlen chunked lengths")
    masked = slice(int(cu_q[3]), int(cu_q[4]))             # queries with no KV rows
    assert torch.all(lse[masked] == -float("inf")) and torch.all(out[masked] == 0)


def test_varlen_config_all_tokens(smla):
    """16384 packed tokens (8192, 4096, 2048, 1024, 1024), h = 64: every
    token against the oracle (host cores), with the tight check."""
    case = mi.config(4)
    d = lambda t: t.to(DEV)
    out, lse = smla.sparse_mla_fwd_varlen(d(case.q), d(case.kv), d(case.indices), d(case.cu_seqlens_q),
                                          d(case.cu_seqlens_kv), case.sm_scale)
    _check_whole("config 4 packed varlen prefill", "varlen", case.q, case.kv, case.indices, out, lse,
                 case.sm_scale, extra={"cu_q": case.cu_seqlens_q, "cu_k": case.cu_seqlens_kv})


def test_varlen_indices_outside_own_sequence(smla):
    """Local indices past a sequence's end land, unmasked, in the next
    sequence's first rows; negative ones other than -1 land in the previous
    sequence's last rows.  Those rows are NaN (and no list of their own
    sequence references them), the rows past the last sequence are NaN, so a
    mapping that fails to mask reads NaN."""
    lens = [300, 200, 257, 130]
    case = mi.varlen_case(630, lens, 8, topk=256)
    cu = [0] + np.cumsum(lens).tolist()
    idx = case.indices.clone()
    g = torch.Generator().manual_seed(631)
    k = 5
    poison = []
    for b in range(len(lens)):
        a, e = cu[b], cu[b + 1]
        L = lens[b]
        own = idx[a:e]
        # no list of a sequence names its own first k or last k positions (poisoned below)
        own[(own >= 0) & (own < k)] = -1
        own[(own >= L - k) & (own < L)] = -1
        # every 9th entry of every 3rd token: past the end (L .. L+k-1) or below -1 (-k-1 .. -2)
        for t in range(0, e - a, 3):
            cols = torch.arange(t % 9, idx.shape[1], 9)
            far = L + torch.randint(0, k, (cols.numel(),), generator=g, dtype=torch.int32)
            neg = -2 - torch.randint(0, k, (cols.numel(),), generator=g, dtype=torch.int32)
            own[t, cols] = torch.where(torch.arange(cols.numel()) % 2 == 0, far, neg)
        poison += list(range(a, a + k)) + list(range(e - k, e))
    total, guard = cu[-1], 64
    # NaN guard rows before the first and after the last sequence
    kv_buf = torch.full((guard + total + guard, 576), float("nan")).to(torch.bfloat16)
    kv = kv_buf[guard:guard + total]
    kv[:] = case.kv
    kv[torch.tensor(poison)] = float("nan")
    d_kv = kv_buf.to(DEV)
    d = lambda t: t.to(DEV)
    out, lse = smla.sparse_mla_fwd_varlen(d(case.q), d_kv[guard:guard + total], d(idx), d(case.cu_seqlens_q),
                                          d(case.cu_seqlens_kv), case.sm_scale)
    counts = smla.debug_valid_count_varlen(d(idx), d(case.cu_seqlens_q), d(case.cu_seqlens_kv), total)
    torch.cuda.synchronize()
    ref_o, ref_l = orc.sparse_mla_fwd_varlen(case.q, kv, idx, case.cu_seqlens_q, case.cu_seqlens_kv,
                                             case.sm_scale)
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "varlen outside own sequence")
    ref_c = orc.valid_count_varlen(idx, case.cu_seqlens_q, case.cu_seqlens_kv)
    assert np.array_equal(counts.cpu().numpy(), ref_c)
    assert ref_c.sum() < int((idx >= 0).sum())   # some non-negative entries really are masked


# ---------------------------------------------------------------- paged decode

def _check_decode(smla, case, tokens=None):
    d = lambda t: t.to(DEV)
    out, lse = smla.sparse_mla_decode(d(case.q), d(case.kv_cache), d(case.block_table), d(case.cache_seqlens),
                                      d(case.indices), case.sm_scale, case.page_size)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy().reshape(-1, case.h_q, 512)
    l = lse.cpu().numpy().reshape(-1, case.h_q)
    ref_o, ref_l = orc.sparse_mla_decode(case.q, case.kv_cache, case.block_table, case.cache_seqlens,
                                         case.indices, case.sm_scale, case.page_size)
    return compare(o, l, ref_o, ref_l, case.name)


def test_decode_small(smla):
    case = mi.decode_case(601, batch=3, s_next=2, h_q=8, lo=100, hi=900, topk=256, page=64, spare_pages=4)
    _check_decode(smla, case)


def test_decode_page16_wide_heads(smla):
    case = mi.decode_case(602, batch=2, s_next=3, h_q=64, lo=50, hi=400, topk=192, page=16, spare_pages=3)
    _check_decode(smla, case)


@pytest.mark.parametrize("h_q,topk,page", [(1, 200, 16), (2, 72, 64), (24, 1000, 16), (128, 136, 32)])
def test_decode_ragged_lists_small_pages(smla, h_q, topk, page):
    """Lists whose last 64-entry block is partial, pages smaller than a
    block, and head counts at the edges of the 16-, 32- and 64-head tiles
    (128: two head groups)."""
    case = mi.decode_case(610 + h_q, batch=3, s_next=2, h_q=h_q, lo=50, hi=1500, topk=topk, page=page,
                          spare_pages=5)
    _check_decode(smla, case)


def test_decode_one_token_cut_over_many_ctas(smla):
    """A single decode token: its 32 blocks are spread over many CTAs, each
    leaving a partial result, and merged."""
    case = mi.decode_case(604, batch=1, s_next=1, h_q=8, lo=9000, hi=9001, topk=2048, spare_pages=2)
    _check_decode(smla, case)


def test_decode_two_head_groups_mostly_empty_pieces(smla):
    """h_q = 128 (two 64-head units per token) over short caches: most of
    each list is -1, so most CTAs' pieces hold no valid entry (empty partials
    with LSE = -inf) and a unit's pieces mix empty and full ones."""
    case = mi.decode_case(605, batch=3, s_next=2, h_q=128, lo=2, hi=200, topk=2048, page=16, spare_pages=2)
    _check_decode(smla, case)


def test_prefill_several_units_per_cta_with_empty_lists(smla):
    """More tokens than SMs, so each CTA runs several units back to back
    (reusing Q and its output staging in turn); every third list is empty."""
    case = mi.prefill_case(406, s_q=700, s_kv=900, h_q=64, topk=256)
    idx = case.indices.clone()
    idx[::3] = -1
    kv = mi.poison_unreferenced(case.kv, torch.unique(idx[idx >= 0]))
    o, l = _run_fwd(smla, case, kv, idx)
    ref_o, ref_l = orc.sparse_mla_fwd(case.q, kv, idx, case.sm_scale)
    compare(o, l, ref_o, ref_l, "several units per CTA")
    assert np.all(o[::3] == 0.0) and np.all(np.isneginf(l[::3]))


def test_decode_dirty_workspace(smla):
    """The workspace arrives with arbitrary contents (here every byte 0xFF):
    a call may read nothing from it that it did not write itself.  Run twice
    on the same buffer."""
    case = mi.decode_case(603, batch=16, s_next=6, h_q=8, lo=4096, hi=9000, topk=2048, spare_pages=4)
    need = smla.decode_workspace_size(case.batch, case.s_next, case.h_q, case.indices.shape[-1])
    assert need > 0, "this shape is expected to split the top-k list"
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)
    d = lambda t: t.to(DEV)
    args = (d(case.q), d(case.kv_cache), d(case.block_table), d(case.cache_seqlens), d(case.indices),
            case.sm_scale, case.page_size)
    ref_o, ref_l = orc.sparse_mla_decode(case.q, case.kv_cache, case.block_table, case.cache_seqlens,
                                         case.indices, case.sm_scale, case.page_size)
    for _ in range(2):
        out, lse = smla.sparse_mla_decode(*args, workspace=ws)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy().reshape(-1, case.h_q, 512)
        l = lse.cpu().numpy().reshape(-1, case.h_q)
        compare(o, l, ref_o, ref_l, "dirty workspace")



def test_decode_concurrent_streams_separate_workspaces(smla):
    """Two decode calls in flight at once on two streams, each with its own
    workspace (its own partials and merge counters): each result equals the
    same call run alone, bit for bit."""
    d = lambda t: t.to(DEV)
    cases = [mi.decode_case(606 + i, batch=8, s_next=6, h_q=8, lo=3000, hi=9000, topk=2048, spare_pages=4)
             for i in range(2)]
    args, refs, wss, outs = [], [], [], []
    for c in cases:
        a = (d(c.q), d(c.kv_cache), d(c.block_table), d(c.cache_seqlens), d(c.indices), c.sm_scale, c.page_size)
        need = smla.decode_workspace_size(c.batch, c.s_next, c.h_q, c.indices.shape[-1])
        assert need > 0, "this shape is expected to split the top-k lists"
        ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)
        refs.append(smla.sparse_mla_decode(*a, workspace=ws))
        torch.cuda.synchronize()
        args.append(a)
        wss.append(ws)
        outs.append((torch.empty_like(refs[-1][0]), torch.empty_like(refs[-1][1])))
    streams = [torch.cuda.Stream(device=DEV) for _ in cases]
    for rep in range(4):
        for i, st in enumerate(streams):
            smla.sparse_mla_decode(*args[i], workspace=wss[i], out=outs[i][0], lse=outs[i][1],
                                   stream=st)
        torch.cuda.synchronize()
        for i in range(len(cases)):
            assert torch.equal(outs[i][0], refs[i][0]) and torch.equal(outs[i][1], refs[i][1]), \
                f"stream {i}, repetition {rep}: differs from the call run alone"
    # and the first result against the oracle
    c = cases[0]
    ref_o, ref_l = orc.sparse_mla_decode(c.q, c.kv_cache, c.block_table, c.cache_seqlens, c.indices, c.sm_scale,
                                         c.page_size)
    compare(outs[0][0].float().cpu().numpy().reshape(-1, c.h_q, 512), outs[0][1].cpu().numpy().reshape(-1, c.h_q),
            ref_o, ref_l, "concurrent decode")

def test_decode_config_all_tokens(smla):
    """batch 16 x 6 MTP tokens, contexts U[4096, 32768], 64-token pages in a
    shuffled pool with every unread slot NaN, h = 8, topk = 2048; every
    token, with the tight check (every list holds 2048 valid entries)."""
    c = mi.config(5)
    d = lambda t: t.to(DEV)
    out, lse = smla.sparse_mla_decode(d(c.q), d(c.kv_cache), d(c.block_table), d(c.cache_seqlens),
                                      d(c.indices), c.sm_scale, c.page_size)
    n = c.batch * c.s_next
    _check_whole("config 5 paged decode", "paged", c.q.reshape(n, c.h_q, 576),
                 c.kv_cache.reshape(-1, 576), c.indices.reshape(n, -1), out.reshape(n, c.h_q, 512),
                 lse.reshape(n, c.h_q), c.sm_scale,
                 extra={"table": c.block_table, "lens": c.cache_seqlens, "page": c.page_size,
                        "num_blocks": c.kv_cache.shape[0], "s_next": c.s_next})


def test_decode_invalid_pages_short_table_and_lengths(smla):
    """Entries the paged mapping must mask although they are non-negative:
    positions past cache_seqlens, pages at or past the table's width
    (max_blocks), table entries -1, -2, num_blocks + 1 and num_blocks + 3.
    The pool sits inside a larger buffer whose pages before and after it are
    NaN, and the table is followed in memory by entries that name a NaN page:
    a mapping that failed to mask would read NaN (or, for a page past the
    width of an earlier request, the next request's pages, which the exact
    valid count catches)."""
    c = mi.decode_case(620, batch=4, s_next=3, h_q=8, lo=400, hi=1000, topk=512, page=64, spare_pages=4)
    nb, page = c.kv_cache.shape[0], c.page_size
    W = 5
    bt = c.block_table[:, :W].clone()
    bt[0, 1] = -1
    bt[1, 0] = -2
    bt[2, 3] = nb + 1
    bt[3, 2] = nb + 3
    lens = c.cache_seqlens.clone()
    lens[1] -= 50
    pre, post = 2, 4
    pool = torch.full((pre + nb + post, page, 576), float("nan")).to(torch.bfloat16)
    pool[pre:pre + nb] = c.kv_cache
    tb = torch.full((c.batch * W + 64,), nb + 1, dtype=torch.int32)
    tb[: c.batch * W] = bt.flatten()
    d_pool, d_tb = pool.to(DEV), tb.to(DEV)
    kv_view = d_pool[pre:pre + nb]
    bt_view = d_tb[: c.batch * W].view(c.batch, W)
    d = lambda t: t.to(DEV)
    out, lse = smla.sparse_mla_decode(d(c.q), kv_view, bt_view, d(lens), d(c.indices), c.sm_scale, page)
    counts = smla.debug_valid_count_paged(d(c.indices), bt_view, d(lens), page, nb)
    torch.cuda.synchronize()
    ref_o, ref_l = orc.sparse_mla_decode(c.q, c.kv_cache, bt, lens, c.indices, c.sm_scale, page)
    compare(out.float().cpu().numpy().reshape(-1, c.h_q, 512), lse.cpu().numpy().reshape(-1, c.h_q),
            ref_o, ref_l, "decode invalid pages")
    ref_c = orc.valid_count_paged(c.indices, bt, lens, page, nb)
    assert np.array_equal(counts.cpu().numpy(), ref_c)
    assert ref_c.sum() < int((c.indices >= 0).sum()) // 2   # most entries are masked here


# ---------------------------------------------------------------- masked set: exact valid counts

def test_debug_valid_count_configs(smla):
    """The debug export (the forward's own gather walk, counting) equals the
    oracle's |V_t| exactly for every token of all five workloads."""
    d = lambda t: t.to(DEV)
    for n in (1, 2, 3):
        c = mi.config(n)
        got = smla.debug_valid_count(d(c.indices), c.kv.shape[0]).cpu().numpy()
        assert np.array_equal(got, orc.valid_count_dense(c.indices, c.kv.shape[0])), f"config {n}"
    c = mi.config(4)
    got = smla.debug_valid_count_varlen(d(c.indices), d(c.cu_seqlens_q), d(c.cu_seqlens_kv), c.kv.shape[0])
    assert np.array_equal(got.cpu().numpy(), orc.valid_count_varlen(c.indices, c.cu_seqlens_q, c.cu_seqlens_kv))
    c = mi.config(5)
    got = smla.debug_valid_count_paged(d(c.indices), d(c.block_table), d(c.cache_seqlens), c.page_size,
                                       c.kv_cache.shape[0])
    ref = orc.valid_count_paged(c.indices, c.block_table, c.cache_seqlens, c.page_size, c.kv_cache.shape[0])
    assert np.array_equal(got.cpu().numpy(), ref)


def test_debug_valid_count_masking_entries(smla):
    """Dense lists mixing -1, other negatives, values at and past s_kv,
    duplicates, ragged list ends (topk not a multiple of 64) and lists longer
    than one 32-block scan window."""
    s_q, s_kv, topk = 40, 700, 2500
    g = torch.Generator().manual_seed(640)
    idx = torch.randint(-800, 1500, (s_q, topk), generator=g, dtype=torch.int32)
    idx[0] = -1
    idx[1, :] = 699
    idx[2, : topk - 1] = -1
    idx[3, ::7] = s_kv
    got = smla.debug_valid_count(idx.to(DEV), s_kv).cpu().numpy()
    ref = orc.valid_count_dense(idx, s_kv)
    assert np.array_equal(got, ref) and ref[0] == 0 and ref[1] == topk


# ---------------------------------------------------------------- determinism

def test_repeated_runs_are_bit_identical(smla):
    """The kernel's reduction order is fixed, so repeated calls on the same
    inputs must agree bit for bit; a copy read by the tensor core before it
    became visible would show up here as run-to-run differences.  Runs are
    interleaved with L2 flushes and decode calls to vary the timing."""
    case = mi.config(2)
    d = lambda t: t.to(DEV)
    q, kv, idx = d(case.q), d(case.kv), d(case.indices)
    dec = mi.decode_case(901, batch=4, s_next=6, h_q=8, lo=3000, hi=9000, topk=2048, spare_pages=4)
    dq, dc, dbt, dsl, di = (d(dec.q), d(dec.kv_cache), d(dec.block_table), d(dec.cache_seqlens), d(dec.indices))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=DEV)
    ref_o, ref_l = smla.sparse_mla_fwd(q, kv, idx, case.sm_scale)
    ref_do, ref_dl = smla.sparse_mla_decode(dq, dc, dbt, dsl, di, dec.sm_scale, dec.page_size)
    for it in range(12):
        if it % 3 == 0:
            flush.zero_()
        o, l = smla.sparse_mla_fwd(q, kv, idx, case.sm_scale)
        do, dl = smla.sparse_mla_decode(dq, dc, dbt, dsl, di, dec.sm_scale, dec.page_size)
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l), f"prefill run {it} differs"
        assert torch.equal(do, ref_do) and torch.equal(dl, ref_dl), f"decode run {it} differs"
    torch.cuda.synchronize()


# ---------------------------------------------------------------- failure detection

def test_device_wait_timeout_reports_and_recovers(smla):
    """A 1 ns bound on device waits makes the kernel give up: it records a
    code, drains, frees TMEM and returns; the host reads the code, clears it
    and the next call is correct."""
    case = mi.prefill_case(701, s_q=16, s_kv=600, h_q=8, topk=512)
    try:
        smla.set_wait_timeout_ns(1)
        _run_fwd(smla, case)
        code = smla.get_device_error()
    finally:
        smla.set_wait_timeout_ns(0)
    assert code != 0 and (code & 0xff) == 1
    smla.clear_device_error()
    assert smla.get_device_error() == 0
    _check_fwd(smla, case)
