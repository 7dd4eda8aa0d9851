"""Comparison of CUDA-path outputs with the oracle (tolerances written here).

Tolerances (per element), against the oracle's result rounded to the I/O type:
  bf16  : at most 1 ulp apart (sign-magnitude ordinals; +0 and -0 are equal)
  fp32  : |y - y_ref| <= 2e-6 * |y_ref|  (y_ref == 0 requires y == 0)
  residual_out : bit-exact
NaN must sit at the same positions on both sides.

Derivation of the fp32 bound: the kernels sum squares in fp32 along a fixed
tree at most 21 levels deep (<= 8 chunk steps, 3 levels over a chunk's
lanes, 5 shuffle levels, 5 levels across warps), a relative error <= 21 u
(u = 2^-24) on the sum, i.e. <= 10.5 u on the scale after the square root;
the mean and eps add 3 roundings (<= 1.5 u on the scale), rsqrtf <= 2 ulp
(<= 4 u), and the two products 2 u: about 18 u = 1.1e-6 relative in the
worst case, inside 2e-6.  A bf16 result computed that accurately is within
one bf16 ulp of the correctly rounded value.
"""
from __future__ import annotations

import numpy as np

F32_RTOL = 2e-6
BF16_MAX_ULP = 1


def bf16_ordinals(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_is_nan(bits):
    b = np.asarray(bits, dtype=np.uint16)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def compare_y(got, ref, dtype):
    """Return (ok, report dict) for a CUDA result against the oracle's."""
    got = np.asarray(got)
    ref = np.asarray(ref)
    if got.shape != ref.shape:
        return False, {"error": f"shape {got.shape} != {ref.shape}"}
    if dtype == "bf16":
        gn, rn = bf16_is_nan(got), bf16_is_nan(ref)
        d = np.abs(bf16_ordinals(got) - bf16_ordinals(ref))
        d = np.where(gn | rn, 0, d)
        nan_ok = np.array_equal(gn, rn)
        worst = int(d.max()) if d.size else 0
        ok = nan_ok and worst <= BF16_MAX_ULP
        return ok, {"max_ulp": worst, "n_1ulp": int((d == 1).sum()), "nan_ok": nan_ok,
                    "n": int(d.size)}
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    gn, rn = np.isnan(g), np.isnan(r)
    nan_ok = np.array_equal(gn, rn)
    with np.errstate(invalid="ignore"):
        both_inf = np.isinf(r) & (g == r)
        err = np.where(gn | rn | both_inf, 0.0, np.abs(g - r))
        lim = F32_RTOL * np.abs(np.where(gn | rn | both_inf, 0.0, r))
    bad = err > lim
    rel = np.where(r != 0, err / np.where(r != 0, np.abs(r), 1.0), np.where(err > 0, np.inf, 0.0))
    worst = float(rel.max()) if rel.size else 0.0
    return nan_ok and not bad.any(), {"max_rel": worst, "n_bad": int(bad.sum()), "nan_ok": nan_ok,
                                      "n": int(r.size)}


def bits_equal(a, b):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    return a.shape == b.shape and a.view(np.uint8).tobytes() == b.view(np.uint8).tobytes()


# LayerNorm: y = w * n + b can cancel, so a relative bound per element does not
# hold; the bound is on the terms instead.  The kernels form the mean and the
# centred sum of squares along fixed trees at most 21 levels deep, so
#   |n' - n| <= 18u |n| + 21u mean|h| / sigma      (sigma = sqrt(var + eps))
# and the fused multiply-add of the output adds u |y|:
#   |y' - y| <= 2e-6 * ( |w| (|n| + mean|h| / sigma) + |b| )
# before the final rounding to the I/O type, which adds at most half an ulp of
# the stored value.
LN_TERM_TOL = 2e-6


def _half_ulp(vals, dtype):
    v = np.abs(vals.astype(np.float64))
    p = 8 if dtype == "bf16" else 24
    qmin = -133 if dtype == "bf16" else -149
    _, e = np.frexp(np.where(v > 0, v, 1.0))
    q = np.maximum(e - p, qmin)
    return np.ldexp(0.5, q)


def decode(a, dtype):
    a = np.asarray(a)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def compare_ln(got, y64, n64, w, b, mean_abs_h, sigma, dtype):
    """CUDA LayerNorm output against the oracle's fp64 value with the term bound above."""
    g = decode(got, dtype)
    wv = np.ones_like(y64) if w is None else decode(w, dtype)[None, :]
    bv = np.zeros_like(y64) if b is None else decode(b, dtype)[None, :]
    bound = LN_TERM_TOL * (np.abs(wv) * (np.abs(n64) + (mean_abs_h / sigma)[:, None]) + np.abs(bv))
    lim = bound + _half_ulp(g, dtype)
    gn, rn = np.isnan(g), np.isnan(y64)
    with np.errstate(invalid="ignore"):
        err = np.where(gn | rn, 0.0, np.abs(g - y64))
    bad = err > lim
    nan_ok = np.array_equal(gn, rn)
    ratio = float((err / np.where(lim > 0, lim, 1)).max()) if err.size else 0.0
    return nan_ok and not bad.any(), {"worst_err_over_bound": ratio, "n_bad": int(bad.sum()), "nan_ok": nan_ok,
                                      "n": int(err.size)}
