"""Comparison helpers for GPU-vs-oracle parity.

Tolerances: bf16 output |g - r| <= 2e-2 + 2e-2 |r| elementwise (the
allclose form of atol=rtol=2e-2, "feat: add XTuner TileLang sparse MLA
backend", Performance); fp32 LSE |g - r| <= 1e-3 absolute; a -inf LSE must
be -inf on both sides and its output row exactly +0.
"""
import numpy as np

ATOL = 2e-2
RTOL = 2e-2
LSE_ATOL = 1e-3


def compare(out_gpu, lse_gpu, ref_out, ref_lse, what=""):
    o = np.asarray(out_gpu, dtype=np.float64)
    l = np.asarray(lse_gpu, dtype=np.float64)
    ref_out = np.asarray(ref_out, dtype=np.float64)
    ref_lse = np.asarray(ref_lse, dtype=np.float64)
    assert o.shape == ref_out.shape, (o.shape, ref_out.shape)
    assert l.shape == ref_lse.shape, (l.shape, ref_lse.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    neg = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), neg), f"{what}: -inf LSE pattern differs"
    if neg.any():
        rows = o[neg]
        assert np.all(rows == 0.0) and not np.any(np.signbit(rows)), f"{what}: masked rows not +0"
    fin = ~neg
    dl = np.abs(l[fin] - ref_lse[fin])
    assert np.all(dl <= LSE_ATOL), f"{what}: max |dlse| = {dl.max():.3e}"
    do = np.abs(o - ref_out)
    bad = do > ATOL + RTOL * np.abs(ref_out)
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs out of tolerance, "
                           f"max |dout| = {do.max():.3e}")
    return float(do.max()), float(dl.max()) if dl.size else 0.0
