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


# Parity statistics of this test session (name -> dict), printed in the
# pytest terminal summary beside the pages' own maximum differences
# ("feat: add XTuner TileLang sparse MLA backend", Performance: 1.22e-4 and
# 2.44e-4 for the two isolated-forward shapes on H200).
RECORD = {}


def record(name, **stats):
    RECORD[name] = stats


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


# A tighter forward check, derived from the kernel's arithmetic, for the
# tokens where the allclose bar above is blind (full 2048-entry lists: one
# dropped row moves an output by far less than 2e-2).  Per element:
#  * out is the bf16 rounding of an fp32 value x: |out - x| <= ulp_bf16(r)
#    (half an ulp of x, and x is within a binade of r);
#  * P is rounded to bf16 before P.V, a relative error delta_j <= 2^-9 per
#    row, independent between rows, variance <= 2^-16 / 12: x - r =
#    sum_j p_j delta_j v_jd has standard deviation
#    sigma_d <= 2^-9 / sqrt(3) * sqrt(sum_j p_j^2 v_jd^2), and the check
#    allows 8 sigma;
#  * the fp32 sums (576-term scores, 2048-term P.V and row sum) add
#    ~1e-6 relative; TIGHT_ATOL covers them.
# A kernel that drops one gathered row's contribution moves the elements of
# that row's largest |v| by p_j |v_jd| (~1e-3 for a typical row of a full
# list), well above this bound.
TIGHT_SIGMAS = 8.0
TIGHT_ATOL = 2e-5


def ulp_bf16(x):
    """Spacing of bf16 numbers at |x| (2^(e - 7) for |x| in [2^e, 2^(e+1)))."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def pv_rounding_sigma(q_t, rows, sm_scale, d_v=512):
    """sigma_d of the P-rounding error (above) for one token: q_t [h, 576],
    rows [n, 576] float64 -> [h, d_v]."""
    q_t = np.asarray(q_t, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    if rows.shape[0] == 0:
        return np.zeros((q_t.shape[0], d_v))
    s = sm_scale * (q_t @ rows.T)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return 2.0 ** -9 / np.sqrt(3.0) * np.sqrt((p * p) @ (rows[:, :d_v] ** 2))


def fp8_rounding_sigma(q_t, rows, sm_scale, d_v=512, d_quant=512):
    """sigma_d for the FP8-cache decode.  At 32 and 64 heads per CTA the
    kernel also rounds every dequantized cache value (the first d_quant
    columns) to bf16 (relative eps_jd, |eps| <= 2^-9, variance <= 2^-16 /
    12) before the products: the score of row j moves by sm_scale * sum_d
    q_d k_jd eps_jd (standard deviation sigma_s_j), the output by sum_j p_j
    [delta_s_j (v_jd - out_d) + v_jd eps_jd], on top of the P rounding of
    pv_rounding_sigma.  At 16 heads the codes enter the products exactly and
    only P times each tile scale is rounded to bf16 (the size of the P
    rounding), so this sigma bounds that arithmetic as well."""
    q_t = np.asarray(q_t, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    if rows.shape[0] == 0:
        return np.zeros((q_t.shape[0], d_v))
    u = 2.0 ** -9 / np.sqrt(3.0)
    s = sm_scale * (q_t @ rows.T)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)                                   # [h, n]
    V = rows[:, :d_v]
    out = p @ V                                                          # [h, d_v]
    sig_s = sm_scale * u * np.sqrt((q_t[:, :d_quant] ** 2) @ (rows[:, :d_quant] ** 2).T)   # [h, n]
    p2 = p * p
    var = 2 * u * u * (p2 @ (V * V))                                     # P rounding + V rounding
    # sum_j p_j^2 sig_s_j^2 (v_jd - out_d)^2, expanded in powers of out_d
    w = p2 * sig_s ** 2
    var += w @ (V * V) - 2 * out * (w @ V) + out * out * w.sum(axis=1, keepdims=True)
    return np.sqrt(np.maximum(var, 0.0))


def tight_ratio(out_gpu, ref_out, sigma):
    """max over elements of |g - r| / (ulp_bf16(r) + 8 sigma + TIGHT_ATOL);
    the tight check passes when this is <= 1."""
    g = np.asarray(out_gpu, dtype=np.float64)
    r = np.asarray(ref_out, dtype=np.float64)
    tol = ulp_bf16(r) + TIGHT_SIGMAS * sigma + TIGHT_ATOL
    return float(np.max(np.abs(g - r) / tol)) if g.size else 0.0


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
