"""Shared comparison helpers for the GPU parity tests (tolerances live here).

Tolerances (stated for bf16 inputs, fp32 accumulation, compared with the fp64
oracle run on the identical bf16 values widened exactly):
  forward / decode:  max |O - O_ref| <= 1e-2, mean |O - O_ref| <= 1e-3,
                     |LSE - LSE_ref| <= 1e-3 on finite entries; -inf where the
                     oracle has -inf (a row that sees no key), with O = 0 there.
  backward:          max |dX - dX_ref| <= 2e-2 * max |dX_ref| for dQ, dK, dV.
These are the stated bounds for the workloads (scale = 1/sqrt(d)).  Off those
workloads, a sharp softmax (large scale) can exceed the fixed 1e-2: P is
rounded to bf16 (relative 2^-9) before the value product and O is rounded to
bf16 at the end, so |O - O_ref| <= 2^-9 max|V| + 2^-9 |O| <= 2^-8 max|V| (plus
fp32 accumulation noise).  ``derived_o_bound`` gives that bound.
"""
import numpy as np
import torch

FWD_MAX_ABS = 1e-2
FWD_MEAN_ABS = 1e-3
LSE_ABS = 1e-3
GRAD_REL = 2e-2


def f64(t):
    """Exact widening of a (bf16 / fp32) tensor to a float64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()


def derived_o_bound(v):
    """Max-abs bound from the arithmetic: two bf16 roundings of weight 2^-9 max|V|."""
    return 2.0 ** -8 * float(np.abs(np.asarray(v, dtype=np.float64)).max()) + 1e-4


def check_out(o, lse, o_ref, lse_ref, what="", max_abs=FWD_MAX_ABS):
    o = np.asarray(o, dtype=np.float64)
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all(), "%s: non-finite output" % what
    assert err.max() <= max_abs, "%s: max |O-O_ref| = %g" % (what, err.max())
    assert err.mean() <= FWD_MEAN_ABS, "%s: mean |O-O_ref| = %g" % (what, err.mean())
    if lse is not None:
        lse = np.asarray(lse, dtype=np.float64)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lse), inf_ref), "%s: -inf LSE pattern differs" % what
        fin = ~inf_ref
        if fin.any():
            le = np.abs(lse[fin] - lse_ref[fin]).max()
            assert le <= LSE_ABS, "%s: max |LSE-LSE_ref| = %g" % (what, le)
    return float(err.max()), float(err.mean())


def check_out_elementwise(o, lse, o_ref, lse_ref, vmax, what=""):
    """Per-element bound for peaked softmaxes, where |O| ~ |v|: the output's
    own bf16 rounding (half an ulp, <= 2^-8 |O|) plus the bf16 rounding of
    the weights before the value product (<= 2^-9 max|V|), plus 1e-4 for
    fp32 accumulation.  The flat max/mean tolerances assume |O| << 1."""
    o = np.asarray(o, dtype=np.float64)
    assert np.isfinite(o).all(), "%s: non-finite output" % what
    bound = 2.0 ** -8 * np.abs(o_ref) + 2.0 ** -9 * vmax + 1e-4
    excess = np.abs(o - o_ref) - bound
    assert excess.max() <= 0, "%s: |O-O_ref| exceeds the rounding bound by %g" % (what, excess.max())
    if lse is not None:
        fin = ~np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(np.asarray(lse)), ~fin), "%s: -inf LSE pattern differs" % what
        if fin.any():
            le = np.abs(np.asarray(lse, dtype=np.float64)[fin] - lse_ref[fin]).max()
            assert le <= LSE_ABS, "%s: max |LSE-LSE_ref| = %g" % (what, le)


def check_out_fp8(o, lse, o_ref, lse_ref, p_ref, v, what=""):
    """FP8 forward against the exact attention of the dequantised inputs, per
    element, with the bound from the arithmetic: P's e4m3 rounding (relative
    2^-4 of each weight, or 2^-10 absolute below 2^-6 in units where the row's
    reference maximum weighs at most 1, i.e. at most max_j P_ij of the
    normalised weight), the bf16 rounding of O (2^-8 |O|), 1e-4 for fp32
    accumulation.  Scores are exact products of e4m3 values accumulated in
    fp32, so the LSE keeps the usual tolerance."""
    o = np.asarray(o, dtype=np.float64)
    assert np.isfinite(o).all(), "%s: non-finite output" % what
    av = np.abs(v)
    bound = (2.0 ** -4 * (p_ref @ av) + 2.0 ** -10 * p_ref.max(axis=-1, keepdims=True) * av.sum(axis=-2, keepdims=True)
             + 2.0 ** -8 * np.abs(o_ref) + 1e-4)
    err = np.abs(o - o_ref)
    excess = (err - bound).max()
    assert excess <= 0, "%s: |O-O_ref| exceeds the FP8 rounding bound by %g" % (what, excess)
    fin = ~np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(np.asarray(lse)), ~fin), "%s: -inf LSE pattern differs" % what
    if fin.any():
        le = np.abs(np.asarray(lse, dtype=np.float64)[fin] - lse_ref[fin]).max()
        assert le <= LSE_ABS, "%s: max |LSE-LSE_ref| = %g" % (what, le)
    return float(err.max()), float(err.mean()), float(bound.mean())


def check_grad(g, g_ref, what="", cancel_scale=None):
    """max |g - g_ref| <= GRAD_REL * max |g_ref|.

    Where the exact gradient vanishes identically (every query sees a single
    key, so dS = P (dP - D) = 0 by cancellation), max |g_ref| is 0 and the
    kernel's result is pure rounding of the cancelling terms; there the error is
    measured against ``cancel_scale`` = scale * max|dP| * max|K or Q|, the size
    of those terms.
    """
    g = np.asarray(g, dtype=np.float64)
    assert np.isfinite(g).all(), "%s: non-finite gradient" % what
    denom = np.abs(g_ref).max()
    if cancel_scale is not None and denom <= 1e-9 * cancel_scale:
        denom = cancel_scale
    rel = np.abs(g - g_ref).max() / max(denom, 1e-30)
    assert rel <= GRAD_REL, "%s: max|dX-ref|/max|ref| = %g" % (what, rel)
    return float(rel)
