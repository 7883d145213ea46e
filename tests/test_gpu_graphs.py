"""The entry points launch asynchronously on the caller's stream, allocate
nothing and never synchronise, so a serving engine can capture them in CUDA
graphs ("feat: add XTuner TileLang sparse MLA backend", Validation: serving
with CUDA graphs).  Each test captures calls with preallocated outputs and
workspaces, replays the graph on new inputs copied into the captured
buffers, and compares the results with direct calls bit for bit (the same
kernels in the same order)."""
import pytest
import torch

import mla_inputs as mi

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def smla(cuda_lib):
    import serving_sparse_mla_gb300 as pkg
    pkg.clear_device_error()
    yield pkg
    assert pkg.get_device_error() == 0


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                      # warm-up outside the graph (first-call setup)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def test_prefill_forward_graph(smla):
    a = mi.prefill_case(701, 300, 300, 8, topk=256)
    b = mi.prefill_case(702, 300, 300, 8, topk=256)
    q, kv, idx = a.q.to(DEV), a.kv.to(DEV), a.indices.to(DEV)
    out = torch.empty((300, 8, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((300, 8), dtype=torch.float32, device=DEV)
    g = _capture(lambda: smla.sparse_mla_fwd(q, kv, idx, a.sm_scale, out=out, lse=lse))
    for case in (b, a):
        q.copy_(case.q)
        kv.copy_(case.kv)
        idx.copy_(case.indices)
        g.replay()
        torch.cuda.synchronize()
        ro, rl = smla.sparse_mla_fwd(case.q.to(DEV), case.kv.to(DEV), case.indices.to(DEV), case.sm_scale)
        torch.cuda.synchronize()
        assert torch.equal(out, ro) and torch.equal(lse, rl)


def test_decode_forward_graph(smla):
    a = mi.decode_case(703, 4, 6, 8, 500, 3000, topk=512, poison=False)
    b = mi.decode_case(703, 4, 6, 8, 500, 3000, topk=512, poison=False)
    b.q.copy_(mi.randn_bf16(mi._gen(704), b.q.shape))
    d = lambda t: t.to(DEV)
    q, kvc, bt, sl, idx = d(a.q), d(a.kv_cache), d(a.block_table), d(a.cache_seqlens), d(a.indices)
    need = smla.decode_workspace_size(4, 6, 8, 512)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=DEV)
    out = torch.empty((4, 6, 8, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((4, 6, 8), dtype=torch.float32, device=DEV)
    g = _capture(lambda: smla.sparse_mla_decode(q, kvc, bt, sl, idx, a.sm_scale, a.page_size, workspace=ws,
                                                out=out, lse=lse))
    q.copy_(b.q)
    g.replay()
    torch.cuda.synchronize()
    ro, rl = smla.sparse_mla_decode(d(b.q), kvc, bt, sl, idx, a.sm_scale, a.page_size)
    torch.cuda.synchronize()
    assert torch.equal(out, ro) and torch.equal(lse, rl)


def test_indexer_graph(smla):
    a = mi.indexer_case(705, 400, 2600, topk=512)
    b = mi.indexer_case(706, 400, 2600, topk=512)
    q, k, w = a.q_idx.to(DEV), a.k_idx.to(DEV), a.weights.to(DEV)
    ws = torch.empty(smla.dsa_indexer_workspace_size(400, 2600, 512), dtype=torch.uint8, device=DEV)
    lst = torch.empty((400, 512), dtype=torch.int32, device=DEV)
    g = _capture(lambda: smla.dsa_indexer_topk(q, k, w, 512, workspace=ws, indices=lst))
    q.copy_(b.q_idx)
    k.copy_(b.k_idx)
    w.copy_(b.weights)
    g.replay()
    torch.cuda.synchronize()
    ref = smla.dsa_indexer_topk(b.q_idx.to(DEV), b.k_idx.to(DEV), b.weights.to(DEV), 512)
    torch.cuda.synchronize()
    assert torch.equal(lst, ref)


def test_dsa_decode_step_graph(smla):
    """One decode step of DSA attention as a single graph: the indexer's
    lists over the paged key cache feed the paged sparse-MLA forward."""
    ic = mi.indexer_paged_case(707, 4, 6, 2500, 6000, topk=1024, poison=False)
    batch, s_next = 4, 6
    g0 = mi._gen(708)
    d = lambda t: t.to(DEV)
    q_idx, k_cache, w = d(ic.q_idx), d(ic.k_cache), d(ic.weights)
    bt, sl = d(ic.block_table), d(ic.cache_seqlens)
    num_blocks, page = ic.k_cache.shape[0], ic.k_cache.shape[1]
    q = d(mi.randn_bf16(g0, (batch, s_next, 8, mi.D_QK)))
    kv_cache = d(mi.randn_bf16(g0, (num_blocks, page, mi.D_QK)))
    max_len = int(ic.cache_seqlens.max())
    ws_i = torch.empty(smla.dsa_indexer_workspace_size(batch * s_next, max_len, 1024), dtype=torch.uint8,
                       device=DEV)
    ws_d = torch.empty(max(smla.decode_workspace_size(batch, s_next, 8, 1024), 16), dtype=torch.uint8, device=DEV)
    lst = torch.empty((batch, s_next, 1024), dtype=torch.int32, device=DEV)
    out = torch.empty((batch, s_next, 8, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((batch, s_next, 8), dtype=torch.float32, device=DEV)
    scale = mi.default_sm_scale()

    def step():
        smla.dsa_indexer_topk_paged(q_idx, k_cache, w, bt, sl, 1024, max_len, workspace=ws_i, indices=lst)
        smla.sparse_mla_decode(q, kv_cache, bt, sl, lst, scale, page, workspace=ws_d, out=out, lse=lse)

    g = _capture(step)
    q_idx.copy_(mi.randn_bf16(mi._gen(709), ic.q_idx.shape))
    q.copy_(mi.randn_bf16(mi._gen(710), q.shape))
    g.replay()
    torch.cuda.synchronize()
    ref_l = smla.dsa_indexer_topk_paged(q_idx, k_cache, w, bt, sl, 1024, max_len)
    ref_o, ref_s = smla.sparse_mla_decode(q, kv_cache, bt, sl, ref_l, scale, page)
    torch.cuda.synchronize()
    assert torch.equal(lst, ref_l)
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_s)
