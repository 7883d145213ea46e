"""sparse_mla_decode_noalloc: paged decode for callers that cannot allocate
device memory at the call (for example a serving engine whose allocator owns
all of HBM after start-up, or a plug-in that only receives device pointers).
It keeps its per-split partial results in a fixed device array inside the
library instead of a caller workspace.

Called through the C ABI, twice in a row on different inputs, it must agree
with sparse_mla_decode given a workspace, and with the float64 oracle, within
the parity tolerances; a shape that needs more scratch than the array holds
is refused before any launch.
"""
import ctypes

import pytest
import torch

import mla_inputs as mi
from oracle import sparse_mla_oracle as orc
from tests.parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
P = lambda t: ctypes.c_void_p(t.data_ptr())


def _upload(case):
    return {k: getattr(case, k).to(DEV) for k in ("q", "kv_cache", "block_table", "cache_seqlens", "indices")}


def _decode(lib, case, d, noalloc, workspace=None):
    b, s, h = case.batch, case.s_next, case.h_q
    out = torch.empty((b, s, h, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((b, s, h), dtype=torch.float32, device=DEV)
    common = (P(d["q"]), P(d["kv_cache"]), P(d["block_table"]), P(d["cache_seqlens"]), P(d["indices"]),
              ctypes.c_float(case.sm_scale), P(out), P(lse), b, s, h, 576, 512, case.indices.shape[-1],
              case.page_size, case.block_table.shape[1], case.kv_cache.shape[0])
    if noalloc:
        st = lib.sparse_mla_decode_noalloc(*common, None)
    else:
        st = lib.sparse_mla_decode(*common, P(workspace), workspace.numel(), None)
    assert st == 0, lib.sparse_mla_status_string(st).decode()
    return out, lse


def test_noalloc_decode_matches_workspace_decode_twice(cuda_lib):
    lib = cuda_lib
    cap = lib.sparse_mla_decode_noalloc_max_scratch_bytes()
    for seed in (801, 802):
        case = mi.decode_case(seed, batch=4, s_next=6, h_q=8, lo=2000, hi=6000, topk=2048, page=64,
                              spare_pages=8)
        need = lib.sparse_mla_decode_workspace_size(case.batch, case.s_next, case.h_q, 512, 2048)
        assert 0 < need <= cap          # the split path, so the scratch array is in use
        d = _upload(case)
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        ref_out, ref_lse = _decode(lib, case, d, noalloc=False, workspace=ws)
        out, lse = _decode(lib, case, d, noalloc=True)
        torch.cuda.synchronize()
        compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out.float().cpu().numpy(),
                ref_lse.cpu().numpy(), f"noalloc seed {seed}")
        ro, rl = orc.sparse_mla_decode(case.q, case.kv_cache, case.block_table, case.cache_seqlens,
                                       case.indices, case.sm_scale, case.page_size)
        compare(out.float().cpu().numpy().reshape(-1, case.h_q, 512), lse.cpu().numpy().reshape(-1, case.h_q),
                ro, rl, f"noalloc seed {seed} vs oracle")


def test_noalloc_decode_refuses_shapes_past_its_scratch(cuda_lib):
    lib = cuda_lib
    batch, s_next, h_q, topk = 1, 4, 64, 8192
    need = lib.sparse_mla_decode_workspace_size(batch, s_next, h_q, 512, topk)
    assert need > lib.sparse_mla_decode_noalloc_max_scratch_bytes()
    # Real device buffers of the call's full extents (all -1 indices), so a
    # call that were wrongly launched could only produce a wrong status or
    # output, never touch memory it does not own.
    q = torch.zeros((batch, s_next, h_q, 576), dtype=torch.bfloat16, device=DEV)
    cache = torch.zeros((8, 64, 576), dtype=torch.bfloat16, device=DEV)
    table = torch.zeros((batch, 8), dtype=torch.int32, device=DEV)
    lens = torch.full((batch,), 64, dtype=torch.int32, device=DEV)
    idx = torch.full((batch, s_next, topk), -1, dtype=torch.int32, device=DEV)
    out = torch.empty((batch, s_next, h_q, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((batch, s_next, h_q), dtype=torch.float32, device=DEV)
    st = lib.sparse_mla_decode_noalloc(P(q), P(cache), P(table), P(lens), P(idx), ctypes.c_float(0.1), P(out),
                                       P(lse), batch, s_next, h_q, 576, 512, topk, 64, 8, 8, None)
    assert st == 6   # SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL, nothing launched
    # argument errors are reported first, with the codes sparse_mla_decode gives
    st = lib.sparse_mla_decode_noalloc(P(q), P(cache), P(table), P(lens), P(idx), ctypes.c_float(0.1), P(out),
                                       P(lse), batch, s_next, h_q, 512, 512, topk, 64, 8, 8, None)
    assert st == 2   # SPARSE_MLA_ERR_UNSUPPORTED_SHAPE (d_qk)
    st = lib.sparse_mla_decode_noalloc(None, P(cache), P(table), P(lens), P(idx), ctypes.c_float(0.1), P(out),
                                       P(lse), batch, s_next, h_q, 576, 512, topk, 64, 8, 8, None)
    assert st == 1   # SPARSE_MLA_ERR_INVALID_ARG (null q)
