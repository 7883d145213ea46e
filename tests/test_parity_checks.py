"""The parity machinery itself, on the CPU: the whole-workload pool and the
tight check of tests/parity.py.  Results that are the oracle's, rounded to
bf16, pass; a result that leaves out one gathered row's P.V contribution
(scores, LSE and normaliser intact) passes the allclose bar of the pages but
fails the tight check."""
import numpy as np
import torch

import mla_inputs as mi
from oracle import sparse_mla_oracle as orc
from tests.oracle_pool import check_all_tokens


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def test_pool_passes_rounded_oracle_dense():
    case = mi.prefill_case(650, s_q=96, s_kv=3000, h_q=8, topk=2048)
    idx = case.indices.clone()
    idx[::8] = torch.stack([torch.randperm(3000, generator=mi._gen(660 + t))[:2048] for t in range(12)]).int()
    ro, rl = orc.sparse_mla_fwd(case.q, case.kv, idx, case.sm_scale)
    st = check_all_tokens("dense", case.q, case.kv, idx, _bf16(ro), torch.from_numpy(rl).float(),
                          case.sm_scale, cores=2, shard_tokens=16)
    assert st["fail"] is None and st["tokens"] == 96
    assert st["tight"] <= 1.0 and st["tight_full"] > 0.0


def test_pool_paged_and_varlen_layouts():
    c = mi.decode_case(651, batch=2, s_next=2, h_q=4, lo=300, hi=600, topk=256, page=64, spare_pages=2)
    ro, rl = orc.sparse_mla_decode(c.q, c.kv_cache, c.block_table, c.cache_seqlens, c.indices, c.sm_scale,
                                   c.page_size)
    n = c.batch * c.s_next
    st = check_all_tokens("paged", c.q.reshape(n, c.h_q, 576), c.kv_cache.reshape(-1, 576),
                          c.indices.reshape(n, -1), _bf16(ro), torch.from_numpy(rl).float(), c.sm_scale,
                          extra={"table": c.block_table, "lens": c.cache_seqlens, "page": c.page_size,
                                 "num_blocks": c.kv_cache.shape[0], "s_next": c.s_next}, cores=2)
    assert st["fail"] is None and st["tokens"] == n and st["tight"] <= 1.0
    v = mi.varlen_case(652, [40, 1, 70], 4, topk=64)
    ro, rl = orc.sparse_mla_fwd_varlen(v.q, v.kv, v.indices, v.cu_seqlens_q, v.cu_seqlens_kv, v.sm_scale)
    st = check_all_tokens("varlen", v.q, v.kv, v.indices, _bf16(ro), torch.from_numpy(rl).float(), v.sm_scale,
                          extra={"cu_q": v.cu_seqlens_q, "cu_k": v.cu_seqlens_kv}, cores=2)
    assert st["fail"] is None and st["tokens"] == v.q.shape[0] and st["tight"] <= 1.0


def test_tight_check_catches_a_dropped_row_the_allclose_bar_misses():
    case = mi.prefill_case(653, s_q=8, s_kv=4000, h_q=8, topk=2048, pattern="recent")
    toks = list(range(8))
    idx = case.indices.clone()
    idx[:, :] = torch.stack([torch.randperm(4000, generator=mi._gen(654 + t))[:2048] for t in toks]).int()
    ro, rl = orc.sparse_mla_fwd(case.q, case.kv, idx, case.sm_scale)
    # leave out the first entry's P.V term of token 3, keeping its LSE
    r = int(idx[3, 0])
    K = case.kv.double().numpy()
    s = case.sm_scale * (case.q[3].double().numpy() @ K[r])
    bad = ro.copy()
    bad[3] -= np.exp(s - rl[3])[:, None] * K[r, :512][None, :]
    st = check_all_tokens("dense", case.q, case.kv, idx, _bf16(bad), torch.from_numpy(rl).float(),
                          case.sm_scale, cores=2)
    assert st["fail"] is None          # within atol = rtol = 2e-2 ...
    assert st["tight"] > 1.0           # ... but not within the tight bound
