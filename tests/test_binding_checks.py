"""Host-side checks of the Python binding (no GPU): the C ABI sees only
pointers and sizes, so the binding refuses, before any launch, a tensor
whose extent is smaller than the sizes it passes imply, a caller-supplied
output of the wrong dtype or layout, and tensors on different devices.
The library is replaced by a recorder and the CUDA-placement test by a
no-op, so the calls run on CPU tensors; valid calls use the shapes of the
GPU parity tests' own cases and must reach the library unchanged."""
import types

import pytest
import torch

import mla_inputs as mi

STREAM = types.SimpleNamespace(cuda_stream=0)


@pytest.fixture
def b(monkeypatch):
    from serving_sparse_mla_gb300 import binding
    calls = []

    class Recorder:
        def __getattr__(self, name):
            def call(*args):
                calls.append(name)
                return 0
            return call

    monkeypatch.setattr(binding, "load", lambda path=None: Recorder())
    monkeypatch.setattr(binding, "_on_cuda", lambda t, name: None)
    binding.calls = calls
    return binding


def _launches(b):
    return [c for c in b.calls if not c.endswith("_workspace_size")]


def _ok(b, entry, fn, *args, **kw):
    del b.calls[:]
    fn(*args, stream=STREAM, **kw)
    assert _launches(b) == [entry]


def _refused(b, fn, *args, match=None, **kw):
    del b.calls[:]
    with pytest.raises(ValueError, match=match):
        fn(*args, stream=STREAM, **kw)
    assert _launches(b) == []


def test_forward_shapes_accepted(b):
    c = mi.prefill_case(1201, s_q=37, s_kv=420, h_q=8, topk=384)
    s_q, h = c.q.shape[:2]
    _ok(b, "sparse_mla_fwd", b.sparse_mla_fwd, c.q, c.kv, c.indices, c.sm_scale)
    _ok(b, "sparse_mla_fwd", b.sparse_mla_fwd, c.q, c.kv.view(420, 1, 576), c.indices.view(s_q, 1, 384), c.sm_scale,
        out=torch.empty((s_q, h, 512), dtype=torch.bfloat16), lse=torch.empty((s_q, h)))
    _ok(b, "sparse_mla_fwd", b.sparse_mla_fwd, c.q[:0], c.kv, c.indices[:0], c.sm_scale)
    _ok(b, "sparse_mla_fwd", b.sparse_mla_fwd, c.q, c.kv[:0], c.indices, c.sm_scale)
    _ok(b, "sparse_mla_fwd_causal", b.sparse_mla_fwd_causal, c.q, c.kv, c.sm_scale)
    v = mi.varlen_case(1260, [130, 1, 257, 64, 40], 8, topk=192)
    _ok(b, "sparse_mla_fwd_varlen", b.sparse_mla_fwd_varlen, v.q, v.kv, v.indices, v.cu_seqlens_q, v.cu_seqlens_kv,
        v.sm_scale)


def test_forward_extents_refused(b):
    c = mi.prefill_case(1201, s_q=37, s_kv=420, h_q=8, topk=384)
    s_q, h = c.q.shape[:2]
    f = b.sparse_mla_fwd
    _refused(b, f, c.q, c.kv, c.indices[:-1], c.sm_scale, match="indices")
    _refused(b, f, c.q, c.kv[:, :512].contiguous(), c.indices, c.sm_scale, match="kv")
    _refused(b, f, c.q, c.kv, c.indices, c.sm_scale, out=torch.empty((s_q - 1, h, 512), dtype=torch.bfloat16),
             match="out")
    _refused(b, f, c.q, c.kv, c.indices, c.sm_scale, lse=torch.empty((s_q, h), dtype=torch.bfloat16), match="lse")
    _refused(b, f, c.q, c.kv, c.indices, c.sm_scale,
             out=torch.empty((h, s_q, 512), dtype=torch.bfloat16).transpose(0, 1), match="contiguous")
    _refused(b, f, c.q, c.kv.to("meta"), c.indices, c.sm_scale, match="kv is on meta")
    _refused(b, b.sparse_mla_fwd_causal, c.q, c.kv, c.sm_scale, out=torch.empty((s_q, h, 256), dtype=torch.bfloat16),
             match="out")
    v = mi.varlen_case(1260, [130, 1, 257, 64, 40], 8, topk=192)
    _refused(b, b.sparse_mla_fwd_varlen, v.q, v.kv, v.indices, v.cu_seqlens_q, v.cu_seqlens_kv[:-1], v.sm_scale,
             match="cu_seqlens_kv")


def test_backward_shapes_and_extents(b):
    c = mi.prefill_case(1210, s_q=29, s_kv=300, h_q=24, topk=256)
    s_q, h = c.q.shape[:2]
    out = torch.zeros((s_q, h, 512), dtype=torch.bfloat16)
    lse = torch.zeros((s_q, h))
    dout = torch.zeros((s_q, h, 512), dtype=torch.bfloat16)
    f = b.sparse_mla_bwd
    _ok(b, "sparse_mla_bwd", f, c.q, c.kv, c.indices, c.sm_scale, out, lse, dout)
    _ok(b, "sparse_mla_bwd", f, c.q, c.kv, c.indices, c.sm_scale, out, lse, dout,
        dq=torch.empty(c.q.shape), dkv=torch.empty((300, 576)))
    _refused(b, f, c.q, c.kv, c.indices, c.sm_scale, out, lse, dout[:-1], match="dout")
    _refused(b, f, c.q, c.kv, c.indices, c.sm_scale, out, lse[:, :8].contiguous(), dout, match="lse")
    _refused(b, f, c.q, c.kv, c.indices, c.sm_scale, out, lse, dout, dkv=torch.empty((299, 576)), match="dkv")
    _refused(b, f, c.q, c.kv, c.indices, c.sm_scale, out, lse, dout, dq=torch.empty(c.q.shape, dtype=torch.bfloat16),
             match="dq")
    v = mi.varlen_case(1264, [130, 1, 257, 64, 40], 64, topk=192)
    t = v.q.shape[0]
    vo, vl, vd = (torch.zeros((t, 64, 512), dtype=torch.bfloat16), torch.zeros((t, 64)),
                  torch.zeros((t, 64, 512), dtype=torch.bfloat16))
    _ok(b, "sparse_mla_bwd_varlen", b.sparse_mla_bwd_varlen, v.q, v.kv, v.indices, v.cu_seqlens_q, v.cu_seqlens_kv,
        v.sm_scale, vo, vl, vd)
    _refused(b, b.sparse_mla_bwd_varlen, v.q, v.kv, v.indices[:-3], v.cu_seqlens_q, v.cu_seqlens_kv, v.sm_scale,
             vo, vl, vd, match="indices")


def test_decode_shapes_and_extents(b):
    c = mi.decode_case(703, 4, 6, 8, 500, 3000, topk=512, poison=False)
    f = b.sparse_mla_decode
    args = (c.q, c.kv_cache, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, c.page_size)
    _ok(b, "sparse_mla_decode", f, *args)
    out = torch.empty((4 * 6, 8, 512), dtype=torch.bfloat16)
    lse = torch.empty((4 * 6, 8))
    _ok(b, "sparse_mla_decode", f, *args, workspace=torch.empty(16, dtype=torch.uint8), out=out.view(4, 6, 8, 512),
        lse=lse.view(4, 6, 8))
    _refused(b, f, c.q, c.kv_cache, c.block_table[:-1], c.cache_seqlens, c.indices, c.sm_scale, c.page_size,
             match="block_table")
    _refused(b, f, c.q, c.kv_cache, c.block_table, c.cache_seqlens[:-1], c.indices, c.sm_scale, c.page_size,
             match="cache_seqlens")
    _refused(b, f, c.q, c.kv_cache, c.block_table, c.cache_seqlens, c.indices[:, :5], c.sm_scale, c.page_size,
             match="indices")
    _refused(b, f, c.q, c.kv_cache, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, 2 * c.page_size,
             match="kv_cache")
    _refused(b, f, *args, out=torch.empty((4, 6, 8, 256), dtype=torch.bfloat16), match="out")
    _refused(b, f, *args, workspace=torch.empty(64, dtype=torch.uint8)[::2], match="contiguous")


def test_fp8_decode_and_debug_count_extents(b):
    c, u = mi.decode_case_fp8(704, 4, 6, 8, 500, 3000, topk=512)
    f = b.sparse_mla_decode_fp8
    args = (c.q, u, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, c.page_size)
    _ok(b, "sparse_mla_decode_fp8", f, *args)
    _refused(b, f, c.q, c.kv_cache, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, c.page_size,
             match="uint8")                                                       # a bf16 cache
    _refused(b, f, c.q, u[..., :576].contiguous(), c.block_table, c.cache_seqlens, c.indices, c.sm_scale, c.page_size,
             match="656")
    _refused(b, f, c.q, u, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, 2 * c.page_size, match="kv_cache")
    _refused(b, f, c.q, u, c.block_table[:-1], c.cache_seqlens, c.indices, c.sm_scale, c.page_size,
             match="block_table")
    _ok(b, "sparse_mla_debug_valid_count_paged", b.debug_valid_count_paged, c.indices, c.block_table,
        c.cache_seqlens, c.page_size, c.kv_cache.shape[0])
    _refused(b, b.debug_valid_count_paged, c.indices, c.block_table[:-1], c.cache_seqlens, c.page_size,
             c.kv_cache.shape[0], match="block_table")
    v = mi.varlen_case(706, [30, 1, 50], 8, topk=64)
    _ok(b, "sparse_mla_debug_valid_count_varlen", b.debug_valid_count_varlen, v.indices, v.cu_seqlens_q,
        v.cu_seqlens_kv, v.kv.shape[0])
    _ok(b, "sparse_mla_debug_valid_count", b.debug_valid_count, v.indices, v.kv.shape[0])


def test_indexer_shapes_and_extents(b):
    c = mi.indexer_case(705, 400, 2600, topk=512)
    q, k, w = c.q_idx, c.k_idx, c.weights
    _ok(b, "dsa_indexer_scores", b.dsa_indexer_scores, q, k, w)
    _ok(b, "dsa_indexer_scores", b.dsa_indexer_scores, q, k, w, row0=50, n_rows=101, skip_len=100)
    _ok(b, "dsa_indexer_topk", b.dsa_indexer_topk, q, k, w, 512)
    _ok(b, "dsa_indexer_topk", b.dsa_indexer_topk, q, k, w, 512, workspace=torch.empty(7 * 2600 * 4, dtype=torch.uint8),
        indices=torch.empty((400, 512), dtype=torch.int32))
    sc = torch.zeros((10, 404))
    _ok(b, "dsa_topk", b.dsa_topk, sc, 64, 30, 400, row0=12, n_rows=10,
        indices=torch.full((30, 64), -7, dtype=torch.int32))
    _refused(b, b.dsa_indexer_scores, q, k, w[:-1], match="weights")
    _refused(b, b.dsa_indexer_scores, q, k[:, :64].contiguous(), w, match="k_idx")
    _refused(b, b.dsa_indexer_scores, q, k, w, n_rows=20, scores=torch.zeros((19, 2600)), match="scores")
    _refused(b, b.dsa_indexer_topk, q, k, w, 512, indices=torch.empty((399, 512), dtype=torch.int32), match="indices")
    _refused(b, b.dsa_topk, sc[:9], 64, 30, 400, row0=12, n_rows=10, match="scores")
    _refused(b, b.dsa_topk, sc, 64, 30, 400, row0=12, n_rows=10, indices=torch.empty((30, 63), dtype=torch.int32),
             match="indices")
    v = mi.indexer_varlen_case(530, [40, 30, 20], [300, 30, 1200], topk=64)
    _ok(b, "dsa_indexer_topk", b.dsa_indexer_topk, v.q_idx, v.k_idx, v.weights, 64, v.cu_seqlens_q, v.cu_seqlens_kv)
    _refused(b, b.dsa_indexer_topk, v.q_idx, v.k_idx, v.weights, 64, v.cu_seqlens_q, v.cu_seqlens_kv[:2],
             match="cu_seqlens_kv")


def test_paged_indexer_shapes_and_extents(b):
    c = mi.indexer_paged_case(707, 4, 6, 2500, 6000, topk=1024, poison=False)
    args = (c.q_idx, c.k_cache, c.weights, c.block_table, c.cache_seqlens)
    _ok(b, "dsa_indexer_topk_paged", b.dsa_indexer_topk_paged, *args, 1024)
    _ok(b, "dsa_indexer_topk_paged", b.dsa_indexer_topk_paged, *args, 1024, max_seqlen_kv=6000,
        indices=torch.empty((4, 6, 1024), dtype=torch.int32), workspace=torch.empty(16, dtype=torch.uint8))
    _ok(b, "dsa_indexer_scores_paged", b.dsa_indexer_scores_paged, *args, 6000)
    _refused(b, b.dsa_indexer_topk_paged, c.q_idx, c.k_cache, c.weights[:, :5], c.block_table, c.cache_seqlens, 1024,
             match="weights")
    _refused(b, b.dsa_indexer_topk_paged, *args, 1024, indices=torch.empty((4, 6, 512), dtype=torch.int32),
             match="indices")
    _refused(b, b.dsa_indexer_scores_paged, *args, 6000, scores=torch.zeros((23, 6000)), match="scores")
    _refused(b, b.dsa_indexer_scores_paged, c.q_idx, c.k_cache[..., :64].contiguous(), c.weights, c.block_table,
             c.cache_seqlens, 6000, match="k_cache")
