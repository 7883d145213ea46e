"""GPU parity of the FP8 KV-cache decode (sparse_mla_decode_fp8) against the
float64 oracle of the dequantized cache (oracle/fp8_kv_oracle.py), on the
same seeded inputs: the allclose bar of the pages on every element, and the
tight bound of tests/parity.py with the FP8 terms (at 32 and 64 heads the
kernel rounds each dequantized value to bf16 before the tensor-core
products; at 16 heads it contracts the codes exactly and rounds P times each
tile scale to bf16)."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
from oracle import fp8_kv_oracle as f8
from oracle import sparse_mla_oracle as orc
from tests.oracle_pool import check_all_tokens
from tests.parity import compare, fp8_rounding_sigma, record, tight_ratio

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def smla(cuda_lib):
    import serving_sparse_mla_gb300 as pkg
    pkg.clear_device_error()
    yield pkg
    assert pkg.get_device_error() == 0


def _run(smla, c, u, **kw):
    d = lambda t: t.to(DEV)
    out, lse = smla.sparse_mla_decode_fp8(d(c.q), d(u), d(c.block_table), d(c.cache_seqlens), d(c.indices),
                                          c.sm_scale, c.page_size, **kw)
    torch.cuda.synchronize()
    return out, lse


def _check(smla, c, u, what):
    out, lse = _run(smla, c, u)
    n = c.batch * c.s_next
    o = out.float().cpu().numpy().reshape(n, c.h_q, 512)
    l = lse.cpu().numpy().reshape(n, c.h_q)
    ro, rl = f8.sparse_mla_decode_fp8(c.q, u, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, c.page_size)
    do, dl = compare(o, l, ro, rl, what)
    # tight bound, token by token
    X = f8.dequantize_slots(u).reshape(-1, 576)
    idx = c.indices.numpy().astype(np.int64)
    tab = c.block_table.numpy().astype(np.int64)
    lens = c.cache_seqlens.numpy()
    worst = 0.0
    for t in range(n):
        b, j = divmod(t, c.s_next)
        r = orc.rows_paged(idx[b, j], tab[b], int(lens[b]), c.page_size, u.shape[0])
        if r.size:
            worst = max(worst, tight_ratio(o[t], ro[t], fp8_rounding_sigma(c.q[b, j].double().numpy(), X[r],
                                                                             c.sm_scale)))
    record(what, max_dout=do, max_dlse=dl, tight_ratio=worst)
    assert worst <= 1.0, f"{what}: tight ratio {worst:.3f}"


@pytest.mark.parametrize("h_q", [8, 24, 64])
def test_fp8_decode_small(smla, h_q):
    c, u = mi.decode_case_fp8(700 + h_q, batch=3, s_next=2, h_q=h_q, lo=100, hi=900, topk=256, page=64,
                              spare_pages=3)
    _check(smla, c, u, f"fp8 decode h={h_q}")


@pytest.mark.parametrize("h_q,topk,page", [(1, 200, 16), (2, 72, 64), (16, 1000, 16), (128, 256, 64)])
def test_fp8_decode_ragged_lists_small_pages(smla, h_q, topk, page):
    """Lists whose last 64-entry block is partial (top-k not a multiple of
    64), pages of 16 rows (a block's rows spread over several pages), one,
    two or sixteen heads in the 16-head tile, and 128 heads (two 64-head
    groups, dequantized in the gather)."""
    c, u = mi.decode_case_fp8(730 + h_q, batch=3, s_next=2, h_q=h_q, lo=50, hi=1500, topk=topk, page=page,
                              spare_pages=5)
    _check(smla, c, u, f"fp8 decode h={h_q} topk={topk} page={page}")


def test_fp8_decode_long_lists_split_over_ctas(smla):
    """One token whose 2048-entry list is cut over many CTAs, and a batch
    whose lists are short (mostly -1) so that many pieces are empty."""
    c, u = mi.decode_case_fp8(711, batch=1, s_next=1, h_q=8, lo=9000, hi=9001, topk=2048, spare_pages=2)
    _check(smla, c, u, "fp8 decode one token")
    c, u = mi.decode_case_fp8(712, batch=3, s_next=2, h_q=16, lo=3, hi=200, topk=2048, page=64, spare_pages=2)
    _check(smla, c, u, "fp8 decode short lists")


@pytest.mark.parametrize("h_q", [24, 64])
def test_fp8_equals_bf16_decode_when_exact(smla, h_q):
    """At 32 and 64 heads per CTA the gather dequantizes each value to bf16
    before the products.  With power-of-two tile scales every dequantized
    value is exact in bf16, so the FP8 decode gathers the very tiles the bf16
    decode gathers from that bf16 cache: the two results agree bit for bit
    (this pins the slot layout: code order, scale of each tile, rope
    offset).  At 16 heads the codes are contracted unscaled (the tile scales
    applied to the partial scores and to P), a different rounding; its
    layout is pinned by the tight bound against the oracle."""
    c, u = mi.decode_case_fp8(713, batch=4, s_next=3, h_q=h_q, lo=500, hi=3000, topk=1024, page=64, spare_pages=2,
                              pow2_scales=True)
    xb = torch.from_numpy(f8.dequantize_slots(u)).to(torch.bfloat16)
    o8, l8 = _run(smla, c, u)
    d = lambda t: t.to(DEV)
    o16, l16 = smla.sparse_mla_decode(d(c.q), d(xb), d(c.block_table), d(c.cache_seqlens), d(c.indices),
                                      c.sm_scale, c.page_size)
    torch.cuda.synchronize()
    assert torch.equal(o8, o16) and torch.equal(l8, l16)


@pytest.mark.parametrize("h_q", [8, 24])
@pytest.mark.parametrize("f", [2.0 ** -20, 2.0 ** 12])
def test_fp8_decode_small_and_large_scales(smla, h_q, f):
    """A cache whose latent values are scaled by a power of two f (tile
    scales from ~1e-8 to ~1e2): the codes are those of the unscaled cache and
    the scales carry f exactly.  The outputs, scaled back by 1/f, must meet
    the tight bound scaled the same way (a relative check: the bound's
    absolute floor would otherwise hide any error at small f), so no
    intermediate of the kernel may under- or overflow at these scales."""
    c, _ = mi.decode_case_fp8(720 + h_q, batch=2, s_next=2, h_q=h_q, lo=300, hi=2000, topk=512, page=64,
                              spare_pages=2)
    c.kv_cache = (c.kv_cache.float() * f).to(torch.bfloat16)
    u = mi.quantize_fp8_slots(c.kv_cache)
    out, lse = _run(smla, c, u)
    n = c.batch * c.s_next
    o = out.float().cpu().numpy().reshape(n, c.h_q, 512)
    l = lse.cpu().numpy().reshape(n, c.h_q)
    ro, rl = f8.sparse_mla_decode_fp8(c.q, u, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, c.page_size)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    X = f8.dequantize_slots(u).reshape(-1, 576)
    idx = c.indices.numpy().astype(np.int64)
    tab = c.block_table.numpy().astype(np.int64)
    lens = c.cache_seqlens.numpy()
    worst = 0.0
    for t in range(n):
        b, j = divmod(t, c.s_next)
        r = orc.rows_paged(idx[b, j], tab[b], int(lens[b]), c.page_size, u.shape[0])
        if r.size:
            qt = c.q[b, j].double().numpy()
            sig = fp8_rounding_sigma(qt, X[r], c.sm_scale)
            worst = max(worst, tight_ratio(o[t] / f, ro[t] / f, sig / f))
            # LSE: moves by at most the largest score error; a score carries
            # at most 2^-9 relative rounding of each dequantized K value
            # (bound taken at 2^-8): sm_scale * 2^-8 * max_j sum_d |q_d k_jd|
            ds = c.sm_scale * 2.0 ** -8 * (np.abs(qt) @ np.abs(X[r]).T).max(axis=1)
            assert np.all(np.abs(l[t] - rl[t]) <= ds + 2e-2), (t, np.abs(l[t] - rl[t]).max(), ds.max())
    record(f"fp8 decode h={h_q}, cache x {f:g}", tight_ratio=worst)
    assert worst <= 1.0, f"cache x {f:g}: relative tight ratio {worst:.3f}"


def test_fp8_decode_config_shape_all_tokens(smla):
    """The paged-decode workload (16 requests x 6 MTP tokens, contexts
    U[4096, 32768], page 64, h = 8, topk = 2048) with its cache in FP8: every
    token against the oracle on the host cores, with the FP8 tight bound."""
    c = mi.config(5)
    u = mi.quantize_fp8_slots(c.kv_cache)
    out, lse = _run(smla, c, u)
    n = c.batch * c.s_next
    st = check_all_tokens("paged_fp8", c.q.reshape(n, c.h_q, 576), u.reshape(-1, 656), c.indices.reshape(n, -1),
                          out.reshape(n, c.h_q, 512).cpu(), lse.reshape(n, c.h_q).cpu(), c.sm_scale,
                          extra={"table": c.block_table, "lens": c.cache_seqlens, "page": c.page_size,
                                 "num_blocks": c.kv_cache.shape[0], "s_next": c.s_next})
    assert st["fail"] is None, st["fail"]
    assert st["tokens"] == n
    record("config 5 paged decode, FP8 cache", tokens=n, max_dout=st["max_dout"], max_dlse=st["max_dlse"],
           tight_ratio=st["tight"])
    assert st["tight"] <= 1.0


def test_fp8_decode_dirty_workspace_twice(smla):
    c, u = mi.decode_case_fp8(714, batch=16, s_next=6, h_q=8, lo=4096, hi=9000, topk=2048, spare_pages=4)
    need = smla.decode_workspace_size(c.batch, c.s_next, c.h_q, 2048)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)
    ro, rl = f8.sparse_mla_decode_fp8(c.q, u, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, c.page_size)
    for _ in range(2):
        out, lse = _run(smla, c, u, workspace=ws)
        compare(out.float().cpu().numpy().reshape(-1, c.h_q, 512), lse.cpu().numpy().reshape(-1, c.h_q), ro, rl,
                "fp8 dirty workspace")
