"""GPU parity of the backward (sparse_mla_bwd through the C ABI) against the
float64 oracle's sparse_mla_bwd on the same seeded inputs.  The forward's
out / lse fed to the backward come from the CUDA forward, as in training."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
from oracle import sparse_mla_oracle as orc
from tests.oracle_pool import oracle_bwd_dense_rows, oracle_fwd_dense_all
from tests.parity import bf16_rounding_err, compare_grad, forward_parity_err, grad_term_bounds, record

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def smla(cuda_lib):
    import serving_sparse_mla_gb300 as pkg
    pkg.clear_device_error()
    yield pkg
    assert pkg.get_device_error() == 0


def _dout(seed, shape):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def _check_bwd(smla, case, idx=None, kv=None, seed=0, what="", cuda_forward=False):
    """The backward is given the oracle forward's out (rounded to bf16) and
    LSE, or with cuda_forward the CUDA forward's, as in training."""
    idx = case.indices if idx is None else idx
    kv = case.kv if kv is None else kv
    dout = _dout(seed, (case.q.shape[0], case.q.shape[1], 512))
    q_d, kv_d, idx_d = case.q.to(DEV), kv.to(DEV), idx.to(DEV)
    if cuda_forward:
        out, lse = smla.sparse_mla_fwd(q_d, kv_d, idx_d, case.sm_scale)
        out_err = forward_parity_err
    else:
        ro, rl = orc.sparse_mla_fwd(case.q, kv, idx, case.sm_scale)
        out = torch.from_numpy(ro).to(torch.bfloat16).to(DEV)
        lse = torch.from_numpy(rl).to(torch.float32).to(DEV)
        out_err = bf16_rounding_err
    dq, dkv = smla.sparse_mla_bwd(q_d, kv_d, idx_d, case.sm_scale, out, lse, dout.to(DEV))
    torch.cuda.synchronize()
    rq, rkv = orc.sparse_mla_bwd(case.q, kv, idx, case.sm_scale, dout)
    bq, bkv = grad_term_bounds(case.q, kv, idx, case.sm_scale, dout, out_err)
    compare_grad(dq.cpu().numpy(), rq, bq, f"{what} dq")
    compare_grad(dkv.cpu().numpy(), rkv, bkv, f"{what} dkv")
    return dq.cpu().numpy(), dkv.cpu().numpy(), rq, rkv


def _check_bwd_sampled(smla, case, dq_tokens, kv_rows, seed, what):
    """Full-size backward (the launch the bench times) checked on sampled
    outputs the oracle computes on its own: dq of the sampled tokens, and dkv
    of the sampled rows, each of which sums the contributions of exactly the
    tokens whose lists hold it (the oracle's backward over those tokens gives
    those rows' full-problem values).  The backward reads the CUDA forward's
    out / LSE for every token, with the oracle's (out rounded to bf16) for the
    tokens the sampled outputs depend on."""
    s_q, h = case.q.shape[0], case.q.shape[1]
    dout = _dout(seed, (s_q, h, 512))
    idx_np = case.indices.numpy()
    listers = np.nonzero(np.isin(idx_np, kv_rows).any(axis=1))[0].tolist()
    need = sorted(set(dq_tokens) | set(listers))
    q_d, kv_d, idx_d = case.q.to(DEV), case.kv.to(DEV), case.indices.to(DEV)
    out, lse = smla.sparse_mla_fwd(q_d, kv_d, idx_d, case.sm_scale)
    ro, rl = orc.sparse_mla_fwd(case.q[need], case.kv, case.indices[need], case.sm_scale)
    sel = torch.tensor(need, dtype=torch.int64, device=DEV)
    out[sel] = torch.from_numpy(ro).to(torch.bfloat16).to(DEV)
    lse[sel] = torch.from_numpy(rl).to(torch.float32).to(DEV)
    dq, dkv = smla.sparse_mla_bwd(q_d, kv_d, idx_d, case.sm_scale, out, lse, dout.to(DEV))
    torch.cuda.synchronize()
    rq, rkv = orc.sparse_mla_bwd(case.q[need], case.kv, case.indices[need], case.sm_scale, dout[need])
    bq, bkv = grad_term_bounds(case.q[need], case.kv, case.indices[need], case.sm_scale, dout[need],
                               bf16_rounding_err)
    pos = {t: i for i, t in enumerate(need)}
    qi = [pos[t] for t in dq_tokens]
    compare_grad(dq[dq_tokens].cpu().numpy(), rq[qi], bq[qi], f"{what} dq (sampled tokens)")
    compare_grad(dkv[kv_rows].cpu().numpy(), rkv[kv_rows], bkv[kv_rows], f"{what} dkv (sampled rows)")
    assert np.all(np.isfinite(dq.cpu().numpy())) and np.all(np.isfinite(dkv.cpu().numpy()))


def test_bwd_small(smla):
    case = mi.prefill_case(1201, s_q=37, s_kv=420, h_q=8, topk=384)
    _check_bwd(smla, case, seed=1, what="small")


@pytest.mark.parametrize("h_q", [1, 16, 24, 64])
def test_bwd_head_counts(smla, h_q):
    """One 16-head unit per token, a ragged second unit (24), four units (64)."""
    case = mi.prefill_case(1210 + h_q, s_q=29, s_kv=300, h_q=h_q, topk=256)
    _check_bwd(smla, case, seed=h_q, what=f"h={h_q}")


def test_bwd_masking_multiplicity_and_unlisted_rows(smla):
    """-1 and out-of-range entries, a row listed several times by one token,
    tokens with no valid entry (dq exactly 0) and rows no token lists (dkv
    exactly 0)."""
    s_q, s_kv, topk = 12, 90, 128
    case = mi.prefill_case(1220, s_q=s_q, s_kv=s_kv, h_q=8, topk=topk)
    g = torch.Generator().manual_seed(1221)
    idx = torch.randint(0, 60, (s_q, topk), generator=g, dtype=torch.int32)   # rows 60.. never listed
    idx[:, ::5] = -1
    idx[:, 3::7] = s_kv + 5
    idx[2, :] = -1                                   # no valid entry
    idx[4, :10] = 7                                  # multiplicity
    dq, dkv, rq, rkv = _check_bwd(smla, case, idx=idx, seed=2, what="masking")
    assert np.all(dq[2] == 0.0)
    assert np.all(dkv[60:] == 0.0)


def test_bwd_full_topk_config1(smla):
    """s_q = s_kv = 64, h = 8, topk = 2048: every causal position listed."""
    _check_bwd(smla, mi.config(1), seed=3, what="config 1")


def test_bwd_long_lists(smla):
    """Lists of 3100 entries (two 32-block scan windows), ragged last block."""
    case = mi.prefill_case(1230, s_q=6, s_kv=5000, h_q=8, topk=3100)
    g = torch.Generator().manual_seed(1231)
    idx = torch.randint(0, 5000, (6, 3100), generator=g, dtype=torch.int32)
    _check_bwd(smla, case, idx=idx, seed=4, what="long lists")


def test_bwd_many_units_per_cta(smla):
    """More token units than SMs: each CTA runs several units in turn."""
    case = mi.prefill_case(1240, s_q=400, s_kv=500, h_q=8, topk=128)
    _check_bwd(smla, case, seed=5, what="several units per CTA")


def test_bwd_after_cuda_forward(smla):
    """Forward then backward on the GPU, as in training: D uses the CUDA
    forward's output, so its error enters through the forward's own bar."""
    case = mi.prefill_case(1250, s_q=60, s_kv=500, h_q=16, topk=256)
    _check_bwd(smla, case, seed=6, what="after CUDA forward", cuda_forward=True)


@pytest.mark.parametrize("h_q", [8, 64])
def test_bwd_varlen(smla, h_q):
    """Packed sequences: local indices into each sequence's own rows; the
    CUDA backward against the oracle's packed backward."""
    case = mi.varlen_case(1260 + h_q, [130, 1, 257, 64, 40], h_q, topk=192)
    d = lambda t: t.to(DEV)
    dout = _dout(h_q, (case.q.shape[0], h_q, 512))
    ro, rl = orc.sparse_mla_fwd_varlen(case.q, case.kv, case.indices, case.cu_seqlens_q, case.cu_seqlens_kv,
                                       case.sm_scale)
    out = torch.from_numpy(ro).to(torch.bfloat16).to(DEV)
    lse = torch.from_numpy(rl).to(torch.float32).to(DEV)
    dq, dkv = smla.sparse_mla_bwd_varlen(d(case.q), d(case.kv), d(case.indices), d(case.cu_seqlens_q),
                                         d(case.cu_seqlens_kv), case.sm_scale, out, lse, d(dout))
    torch.cuda.synchronize()
    rq, rkv = orc.sparse_mla_bwd_varlen(case.q, case.kv, case.indices, case.cu_seqlens_q, case.cu_seqlens_kv,
                                        case.sm_scale, dout)
    cu_q = case.cu_seqlens_q.numpy()
    cu_k = case.cu_seqlens_kv.numpy()

    def rows_of(t, idx_t):
        b = int(np.searchsorted(cu_q, t, side="right") - 1)
        n = int(cu_k[b + 1] - cu_k[b])
        return int(cu_k[b]) + idx_t[(idx_t >= 0) & (idx_t < n)]
    bq, bkv = grad_term_bounds(case.q, case.kv, case.indices, case.sm_scale, dout, bf16_rounding_err,
                               rows_of=rows_of)
    compare_grad(dq.cpu().numpy(), rq, bq, f"varlen h={h_q} dq")
    compare_grad(dkv.cpu().numpy(), rkv, bkv, f"varlen h={h_q} dkv")


def test_bwd_varlen_chunked_lengths_and_empty_sequences(smla):
    """The packed backward with query and KV lengths that differ per
    sequence, an empty sequence, one with KV rows but no queries and one with
    queries but no KV rows (their dq is 0), lists with entries past the
    sequence's KV end (masked) and -1 padding."""
    lens_q = [90, 0, 0, 23, 12, 6]
    lens_kv = [260, 0, 40, 0, 64, 500]
    topk = 192
    g = torch.Generator().manual_seed(1280)
    total_q, total_kv = sum(lens_q), sum(lens_kv)
    q = torch.randn((total_q, 16, 576), generator=g).to(torch.bfloat16)
    kv = torch.randn((total_kv, 576), generator=g).to(torch.bfloat16)
    idx = torch.full((total_q, topk), -1, dtype=torch.int32)
    t = 0
    for lq, lk in zip(lens_q, lens_kv):
        for _ in range(lq):
            n = min(topk - 8, lk)
            if n:
                idx[t, :n] = torch.randperm(lk, generator=g)[:n].to(torch.int32)
            idx[t, n:n + 8] = lk + torch.arange(8, dtype=torch.int32)
            t += 1
    cu_q = torch.tensor([0] + np.cumsum(lens_q).tolist(), dtype=torch.int32)
    cu_kv = torch.tensor([0] + np.cumsum(lens_kv).tolist(), dtype=torch.int32)
    sm_scale = 1.0 / 24.0
    dout = _dout(1281, (total_q, 16, 512))
    ro, rl = orc.sparse_mla_fwd_varlen(q, kv, idx, cu_q, cu_kv, sm_scale)
    d = lambda x: x.to(DEV)
    out = torch.from_numpy(ro).to(torch.bfloat16).to(DEV)
    lse = torch.from_numpy(rl).to(torch.float32).to(DEV)
    dq, dkv = smla.sparse_mla_bwd_varlen(d(q), d(kv), d(idx), d(cu_q), d(cu_kv), sm_scale, out, lse, d(dout))
    torch.cuda.synchronize()
    rq, rkv = orc.sparse_mla_bwd_varlen(q, kv, idx, cu_q, cu_kv, sm_scale, dout)
    cq, ck = cu_q.numpy(), cu_kv.numpy()

    def rows_of(t, idx_t):
        b = int(np.searchsorted(cq, t, side="right") - 1)
        n = int(ck[b + 1] - ck[b])
        return int(ck[b]) + idx_t[(idx_t >= 0) & (idx_t < n)]
    bq, bkv = grad_term_bounds(q, kv, idx, sm_scale, dout, bf16_rounding_err, rows_of=rows_of)
    compare_grad(dq.cpu().numpy(), rq, bq, "varlen chunked dq")
    compare_grad(dkv.cpu().numpy(), rkv, bkv, "varlen chunked dkv")
    assert torch.all(dq[int(cq[3]):int(cq[4])] == 0)      # queries with no KV rows


def test_bwd_mid_prefill_config_sampled(smla):
    """s_q = s_kv = 2119, h = 8, topk = 2048 (16-head units): sampled dq
    tokens and dkv rows listed by 1 to ~120 tokens."""
    g = np.random.default_rng(21)
    toks = sorted(set([0, 1, 127, 128, 2047, 2048, 2118] + g.choice(2119, 13, replace=False).tolist()))
    _check_bwd_sampled(smla, mi.config(2), toks, [2118, 2100, 2030, 2000], seed=21, what="config 2")


def test_bwd_wide_head_config_sampled(smla):
    """s_q = s_kv = 8192, h = 64, topk = 2048 (two 32-head units per token):
    sampled dq tokens and dkv rows listed by 1 to ~170 tokens (the recent
    window and the random tail of the list pattern)."""
    g = np.random.default_rng(31)
    toks = sorted(set([0, 1, 127, 128, 2047, 2048, 4095, 8191] + g.choice(8192, 16, replace=False).tolist()))
    _check_bwd_sampled(smla, mi.config(3), toks, [8191, 8150, 8064, 7900], seed=31, what="config 3")


@pytest.mark.parametrize("cfg", [2, 3])
def test_bwd_heavily_listed_rows_full_size(smla, cfg):
    """dkv rows 0 .. 127 at full size (configs 2 and 3, the launch the bench
    times): almost every token lists them, so each sums ~2000-8000 fp32
    atomic contributions.  The backward is given the oracle forward's out
    (rounded to bf16) and LSE for every token, and its dkv rows are compared
    with the oracle's backward summed over every listing token (host cores)."""
    case = mi.config(cfg)
    rows = list(range(128))
    s_q, h = case.q.shape[0], case.q.shape[1]
    dout = _dout(40 + cfg, (s_q, h, 512))
    out, lse = oracle_fwd_dense_all(case.q, case.kv, case.indices, case.sm_scale)
    dq, dkv = smla.sparse_mla_bwd(case.q.to(DEV), case.kv.to(DEV), case.indices.to(DEV), case.sm_scale,
                                  out.to(DEV), lse.to(DEV), dout.to(DEV))
    torch.cuda.synchronize()
    ref, bound, listers = oracle_bwd_dense_rows(case.q, case.kv, case.indices, dout, case.sm_scale, rows)
    assert listers > 0.9 * s_q
    worst = compare_grad(dkv[rows].cpu().numpy(), ref, bound, f"config {cfg} dkv rows 0..127")
    record(f"config {cfg} backward, dkv rows 0..127", listing_tokens=listers,
           max_ddkv=float(np.abs(dkv[rows].cpu().numpy() - ref).max()), worst_bound_ratio=worst)
    assert np.all(np.isfinite(dq.cpu().numpy()))
