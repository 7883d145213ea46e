"""sparse_mla_decode_noalloc: paged decode for callers that cannot allocate
device memory at the call (for example a serving engine whose allocator owns
all of HBM after start-up, or a plug-in that only receives device pointers).
It keeps its per-split partial results in a fixed device array inside the
library instead of a caller workspace.

Called through the C ABI, twice in a row on different inputs, it must agree
with sparse_mla_decode given a workspace, within the parity tolerances; a
shape that needs more scratch than the array holds is refused before any
launch.
"""
import ctypes

import pytest
import torch

import mla_inputs as mi
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


def test_noalloc_decode_refuses_shapes_past_its_scratch(cuda_lib):
    lib = cuda_lib
    batch, s_next, h_q, topk = 1, 4, 64, 8192
    need = lib.sparse_mla_decode_workspace_size(batch, s_next, h_q, 512, topk)
    assert need > lib.sparse_mla_decode_noalloc_max_scratch_bytes()
    st = lib.sparse_mla_decode_noalloc(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                       ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_float(0.1),
                                       ctypes.c_void_p(16), ctypes.c_void_p(16), batch, s_next, h_q, 576, 512, topk,
                                       64, 8, 8, None)
    assert st == 6   # SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL, nothing launched
