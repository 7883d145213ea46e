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


# Gradients.  Two error sources bound an element of dq / dkv:
#  * the kernel rounds every term's factor sm_scale*dS (and P) to bf16 for the
#    tensor core, relative error <= 2^-9 each: at most 2^-8 * sum |term|;
#  * D = rowsum(dout * out) uses the forward output it is given, not the exact
#    O; with |out - O| <= out_err elementwise, |dD| <= sum_d |dout| out_err,
#    and dS moves by P * dD * sm_scale, so dq moves by at most
#    sm_scale * dD * sum_j P_j |K_j| and dkv rows by sm_scale * dD * P_j |q|.
# grad_term_bounds computes both in float64 from the same inputs; the check is
#   |g - r| <= bound + GRAD_ATOL_RMS * rms(r) + GRAD_RTOL * |r|.
GRAD_RTOL = 2e-2
GRAD_ATOL_RMS = 1e-3


def grad_term_bounds(q, kv, indices, sm_scale, dout, out_err, d_v=512, rows_of=None):
    """Per-element error bounds of dq and dkv (see above).  out_err(O) gives
    the elementwise bound on |out - O| for the forward output the backward
    was given, from the exact O; rows_of(t, idx_t) maps a token's list to KV
    rows (default: the dense layout)."""
    import torch
    f64 = lambda x: x.double().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float64)
    qf, kvf, dof = f64(q), f64(kv), f64(dout)
    idx = indices.numpy() if isinstance(indices, torch.Tensor) else np.asarray(indices)
    s_q, h, d_qk = qf.shape
    s_kv = kvf.shape[0]
    bq = np.zeros_like(qf)
    bkv = np.zeros_like(kvf)
    for t in range(s_q):
        if rows_of is None:
            r = idx[t][(idx[t] >= 0) & (idx[t] < s_kv)].astype(np.int64)
        else:
            r = np.asarray(rows_of(t, idx[t]), dtype=np.int64)
        if r.size == 0:
            continue
        K = kvf[r]
        s = sm_scale * (qf[t] @ K.T)
        P = np.exp(s - s.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        O = P @ K[:, :d_v]
        dP = dof[t] @ K[:, :d_v].T
        D = (dof[t] * O).sum(axis=1, keepdims=True)
        dS = np.abs(sm_scale * P * (dP - D))
        dD = (np.abs(dof[t]) * out_err(O)).sum(axis=1, keepdims=True)      # [h, 1]
        shift = sm_scale * P * dD                                            # |change of dS| per entry
        bq[t] = 2.0 ** -8 * (dS @ np.abs(K)) + shift @ np.abs(K)
        np.add.at(bkv, r, 2.0 ** -8 * (dS.T @ np.abs(qf[t])) + shift.T @ np.abs(qf[t]))
        np.add.at(bkv[:, :d_v], r, 2.0 ** -8 * (P.T @ np.abs(dof[t])))
    return bq, bkv


def bf16_rounding_err(O):
    """|bf16(O) - O| <= 2^-9 |O| (round to nearest even)."""
    return 2.0 ** -9 * np.abs(O)


def forward_parity_err(O):
    """The forward's own bar, |out - O| <= 2e-2 + 2e-2 |O|."""
    return ATOL + RTOL * np.abs(O)


def compare_grad(g, r, bound, what=""):
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite gradient"
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    d = np.abs(g - r)
    tol = bound + GRAD_ATOL_RMS * rms + GRAD_RTOL * np.abs(r)
    bad = d > tol
    i = int(np.argmax(d / np.maximum(tol, 1e-300)))
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {r.size} out of tolerance; worst element "
                           f"|d| = {d.flat[i]:.3e}, bound = {np.asarray(bound).flat[i]:.3e}, "
                           f"rms(ref) = {rms:.3e}")
    return float(np.max(d / np.maximum(tol, 1e-300)))
