"""Comparison of CUDA-path outputs with the oracle (tolerances written here).

Tolerances (per element), against the oracle's result rounded to the I/O type:
  bf16  : at most 1 ulp apart (sign-magnitude ordinals; +0 and -0 are equal)
  fp32  : |y - y_ref| <= 2e-6 * |y_ref|  (y_ref == 0 requires y == 0)
  residual_out : bit-exact
NaN must sit at the same positions on both sides.

Derivation of the fp32 bound: the register and two-pass kernels sum squares
in fp32 along a fixed tree at most 21 levels deep (<= 8 chunk steps, 3 levels
over a chunk's lanes, 5 shuffle levels, 5 levels across warps), a relative
error <= 21 u (u = 2^-24) on the sum, i.e. <= 10.5 u on the scale after the
square root;
the mean and eps add 3 roundings (<= 1.5 u on the scale), rsqrtf <= 2 ulp
(<= 4 u), and the two products 2 u: about 18 u = 1.1e-6 relative in the
worst case, inside 2e-6.  (The bulk-copy kernel's tree is at most 35 levels
deep, 24 chunk steps for fp32 rows of 49152: about 25 u = 1.5e-6, still
inside.  The cluster kernel's tree is at most 21 levels deep too: 8 chunk
steps, 2 lane levels, 5 shuffle levels, 3 warp levels and 3 levels over the
cluster's partial sums for fp32 rows in 32 KB slices.)  A bf16 result
computed that accurately is within one bf16 ulp of the correctly rounded
value.
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


# RMSNorm in the op-by-op cast order, bf16: y = RN(RN(n) * w) with n = h * r.
# The kernel's normalised value n' obeys the fp32 bound above,
# |n' - n| <= CAST_REL_TOL |n|, so RN(n') = RN(n) except where n lies that
# close to a bf16 rounding midpoint; there either neighbour is correct, and y
# must be the weight product (rounded once, exactly as defined) of the one the
# kernel took.  Everything else is bit-exact.
CAST_REL_TOL = F32_RTOL


def compare_cast_bf16(got, n64, w_bits, bf16_from_double):
    """Return (ok, report) for bf16 cast-order outputs against the oracle's
    fp64 normalised values ``n64`` and the weight bits (None: no weight)."""
    got = np.asarray(got, dtype=np.uint16)
    n64 = np.asarray(n64, dtype=np.float64)
    if got.shape != n64.shape:
        return False, {"error": f"shape {got.shape} != {n64.shape}"}
    lo = bf16_from_double(n64 * (1.0 - CAST_REL_TOL)).reshape(n64.shape)
    hi = bf16_from_double(n64 * (1.0 + CAST_REL_TOL)).reshape(n64.shape)
    wv = 1.0 if w_bits is None else decode(w_bits, "bf16")[None, :]
    y_lo = bf16_from_double(decode(lo, "bf16") * wv).reshape(n64.shape)
    y_hi = bf16_from_double(decode(hi, "bf16") * wv).reshape(n64.shape)
    ok = (got == y_lo) | (got == y_hi)
    return bool(ok.all()), {"n_bad": int((~ok).sum()), "n_boundary": int((lo != hi).sum()), "n": int(got.size)}


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


# MXFP8: integers (E4M3 codes, E8M0 scales) decided by floating point.  The
# kernel decides them from its fp32 values of the op, which are within
# MX_REL_TOL (the fp32 bound derived above) of the exact values; a code or a
# scale may therefore differ from the oracle's only where the exact value lies
# that close to the decision boundary.  Everything else must match exactly.
MX_REL_TOL = 2e-6


def _e4m3_values(codes):
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(ef == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * np.ldexp(1.0, ef - 7))
    return np.where((ef == 0xF) & (m == 0x7), np.nan, sign * val)


def compare_mx(codes_g, scales_g, codes_o, scales_o, v64, e4m3_encode):
    """Check GPU MXFP8 output against the oracle's; ``e4m3_encode`` is the
    oracle's encoder (used to re-derive the codes under an alternative scale)."""
    codes_g = np.asarray(codes_g)
    rows, hidden = codes_g.shape
    nb = hidden // 32
    vb = v64.reshape(rows, nb, 32)
    special = ~np.isfinite(vb).all(axis=2)
    amax = np.where(special, 0.0, np.abs(np.where(np.isfinite(vb), vb, 0.0)).max(axis=2))
    sg = np.asarray(scales_g).astype(np.int64)
    so = np.asarray(scales_o).astype(np.int64)
    report = {"scale_flips": 0, "code_flips": 0, "bad": 0}
    # scales: equal, or amax within tolerance of the power of two between them
    diff = sg != so
    if diff.any():
        with np.errstate(divide="ignore"):
            lg = np.log2(np.where(amax > 0, amax, 1.0))
        near = np.abs(lg - np.round(lg)) < MX_REL_TOL * 1.45
        ok_flip = diff & ~special & (np.abs(sg - so) == 1) & near
        report["scale_flips"] = int(ok_flip.sum())
        if (diff & ~ok_flip).any():
            report["bad"] += int((diff & ~ok_flip).sum())
            return False, report
    # expected codes under the GPU's scales
    scaled = vb * np.ldexp(1.0, -(sg - 127))[:, :, None]
    want = e4m3_encode(np.where(np.isfinite(scaled), scaled, 0.0)).reshape(rows, nb, 32)
    want = np.where(special[:, :, None], 0x7F, want)
    got = codes_g.reshape(rows, nb, 32).astype(np.int64)
    mism = got != want
    if mism.any():
        vg = _e4m3_values(got)
        vw = _e4m3_values(want)
        mid = (vg + vw) / 2
        adjacent = np.abs((got & 0x7F) - (want & 0x7F)) == 1
        near = np.abs(scaled - mid) <= MX_REL_TOL * np.abs(scaled)
        sat = (np.abs(scaled) > 448.0) & ((got & 0x7F) == 0x7E)      # saturated either way
        ok = mism & ((adjacent & near) | sat)
        report["code_flips"] = int(ok.sum())
        report["bad"] += int((mism & ~ok).sum())
    return report["bad"] == 0, report


# NVFP4: as MXFP8, integers decided by fp32.  The kernel's block scale comes
# from amax * RN(1 / (6 S)) and its codes from v * rcp(RN(scale * S)) with a
# fast reciprocal (<= 2 ulp): a few 1e-7 more than the exact quotients on top
# of the op's 1.1e-6, inside NV_REL_TOL.
NV_REL_TOL = 2.5e-6
E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e4m3_mid_near(t, a, b, tol):
    """t (>= 0) lies within tol (relative) of the midpoint of E4M3 codes a, b."""
    va, vb = _e4m3_values(a), _e4m3_values(b)
    m = (va + vb) / 2
    return np.abs(t - m) <= tol * np.maximum(m, 1e-300)


def compare_nv(packed_g, scales_g, packed_o, scales_o, v64, tensor_scale, e2m1_encode):
    g = np.asarray(packed_g)
    rows = g.shape[0]
    cg = np.empty((rows, g.shape[1] * 2), dtype=np.int64)
    cg[:, 0::2], cg[:, 1::2] = g & 0xF, g >> 4
    hidden = cg.shape[1]
    nb = hidden // 16
    vb = v64.reshape(rows, nb, 16)
    S = float(np.float32(tensor_scale))
    special = ~np.isfinite(vb).all(axis=2)
    amax = np.where(special, 0.0, np.abs(np.where(np.isfinite(vb), vb, 0.0)).max(axis=2))
    sg = np.asarray(scales_g).astype(np.int64)
    so = np.asarray(scales_o).astype(np.int64)
    rep = {"scale_flips": 0, "code_flips": 0, "bad": 0}
    diff = sg != so
    if diff.any():
        t = amax / (6.0 * S)
        ok_flip = diff & ~special & (np.abs(sg - so) == 1) & _e4m3_mid_near(t, sg, so, NV_REL_TOL)
        rep["scale_flips"] = int(ok_flip.sum())
        if (diff & ~ok_flip).any():
            rep["bad"] += int((diff & ~ok_flip).sum())
            return False, rep
    sv = np.where(special, 0.0, _e4m3_values(sg))
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(sv[:, :, None] > 0, vb / (sv[:, :, None] * S), 0.0)
    want = e2m1_encode(np.where(np.isfinite(scaled), scaled, 0.0)).reshape(rows, nb, 16).astype(np.int64)
    want = np.where(special[:, :, None], 0, want)
    got = cg.reshape(rows, nb, 16)
    mism = got != want
    if mism.any():
        lo = np.minimum(got & 7, want & 7)
        hi = np.maximum(got & 7, want & 7)
        mid = (E2M1_MAGS[lo] + E2M1_MAGS[np.minimum(hi, 7)]) / 2
        adjacent = (hi - lo == 1) & ((got & 8) == (want & 8))
        near = np.abs(np.abs(scaled) - mid) <= NV_REL_TOL * np.maximum(mid, 1e-300)
        ok = mism & adjacent & near
        rep["code_flips"] = int(ok.sum())
        rep["bad"] += int((mism & ~ok).sum())
    return rep["bad"] == 0, rep
