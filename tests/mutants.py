"""Deliberately broken RMSNorm variants, used to show that the pins catch the
plausible mistakes an oracle could make (a dropped term, a wrong index, the
wrong rounding, eps in the wrong place ...).

``reference(...)`` is an independent numpy fp64 restatement of the definition
("Building a GPU compiler from scratch ... (Emmy)", running example and
section "Tensor IR").  With ``mistake=None`` it must pass every pin; with any
named mistake at least one pin must fail.  Test code only.
"""
from __future__ import annotations

import numpy as np

# significant bits, smallest quantum exponent, largest finite value
_FMT = {"bf16": (8, -133, 255.0 * 2.0 ** 120), "f32": (24, -149, (2.0 ** 24 - 1) * 2.0 ** 104)}

MISTAKES = [
    "eps_on_sum", "eps_outside_sqrt", "divide_by_h_minus_1", "no_sqrt", "sqrt_not_inverse",
    "weight_reversed", "no_weight", "unrounded_residual", "global_mean", "trunc_rounding",
    "ties_away", "abs_output", "residual_out_is_x", "sum_of_abs", "stats_from_x",
    "eps_as_double", "round_via_f32",
]
# Planted mistakes of the weight-bias form and of the per-head Q/K layout.
BIAS_MISTAKES = ["bias_ignored", "bias_added_to_output", "bias_scaled_by_r"]
QK_MISTAKES = ["qk_weights_swapped", "qk_one_weight", "qk_stats_over_token", "qk_head_offset"]


def _round(v, dt, mode="rne"):
    """Round fp64 values to the format (value as fp64) with the given tie rule."""
    p, qmin, vmax = _FMT[dt]
    a = np.abs(v)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(a)
        q = np.maximum(e - p, qmin)
        s = np.ldexp(a, -q)
        if mode == "rne":
            n = np.rint(s)
        elif mode == "trunc":
            n = np.floor(s)
        else:  # ties away from zero
            n = np.floor(s + 0.5)
        r = np.ldexp(n, q)
        r = np.where(np.isinf(a), np.inf, r)
        r = np.where(r > vmax, np.inf, r)
        r = np.copysign(r, v)
        r = np.where(np.isnan(v), np.nan, r)
    return r


def _decode(a, dt):
    if dt == "bf16":
        return (np.asarray(a, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _encode(v, dt):
    f = v.astype(np.float32)   # exact: v already holds a value of the format
    if dt == "bf16":
        return (f.view(np.uint32) >> 16).astype(np.uint16)
    return f


def reference(x, w, residual, eps, dt, mistake=None, weight_bias=0.0):
    mode = {"trunc_rounding": "trunc", "ties_away": "away"}.get(mistake, "rne")
    b = float(np.float32(weight_bias or 0.0))
    xv = _decode(x, dt)
    e = float(eps) if mistake == "eps_as_double" else float(np.float32(eps))
    if residual is not None:
        s = xv + _decode(residual, dt)
        h_store = _round(s, dt, mode)
        h = s if mistake == "unrounded_residual" else h_store
        if mistake == "residual_out_is_x":
            h_store = xv
    else:
        h = xv
        h_store = None
    stats = xv if mistake == "stats_from_x" else h
    n = h.shape[1]
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        sq = np.abs(stats) if mistake == "sum_of_abs" else stats * stats
        if mistake == "global_mean":
            total = sq.sum() / sq.size * n
            ssum = np.full((h.shape[0], 1), total)
        else:
            ssum = sq.sum(axis=1, keepdims=True)
        denom = n - 1 if (mistake == "divide_by_h_minus_1" and n > 1) else n
        if mistake == "eps_on_sum":
            inner = ssum + e
            mean_e = inner / denom
        else:
            mean_e = ssum / denom + e
        if mistake == "eps_outside_sqrt":
            r = 1.0 / (np.sqrt(ssum / denom) + e)
        elif mistake == "no_sqrt":
            r = 1.0 / mean_e
        elif mistake == "sqrt_not_inverse":
            r = np.sqrt(mean_e)
        else:
            r = 1.0 / np.sqrt(mean_e)
        y = h * r
        if w is not None and mistake != "no_weight":
            wv = _decode(w, dt)
            if mistake == "weight_reversed":
                wv = wv[::-1]
            if mistake == "bias_added_to_output":
                y = y * wv + b
            elif mistake == "bias_scaled_by_r":
                y = h * (r * wv + b)
            elif mistake == "bias_ignored":
                y = y * wv
            else:
                y = y * (wv + b)
        if mistake == "abs_output":
            y = np.abs(y)
    if mistake == "round_via_f32":
        y = y.astype(np.float32).astype(np.float64)
    yr = _round(y, dt, mode)
    out_y = _encode(yr, dt)
    out_h = None if h_store is None else _encode(h_store, dt)
    return out_y, out_h, y


def reference_qk(x, q_heads, k_heads, head_dim, q_w, k_w, eps, dt, weight_bias=0.0, mistake=None):
    """Per-head Q/K norm of packed token rows built on ``reference``."""
    tokens = x.shape[0]
    qc, kc = q_heads * head_dim, k_heads * head_dim
    if mistake == "qk_head_offset":
        qc_start = head_dim // 2
    else:
        qc_start = 0
    q_rows = np.ascontiguousarray(x[:, qc_start:qc_start + qc]).reshape(tokens * q_heads, head_dim)
    k_rows = np.ascontiguousarray(x[:, qc:qc + kc]).reshape(tokens * k_heads, head_dim)
    qw, kw = (k_w, q_w) if mistake == "qk_weights_swapped" else (q_w, k_w)
    if mistake == "qk_one_weight":
        kw = qw
    if mistake == "qk_stats_over_token":
        both = np.concatenate([x[:, :qc], x[:, qc:qc + kc]], axis=1)
        yall, _, _ = reference(both, None, None, eps, dt)
        # rescale as if a whole-token norm were taken: wrong statistics per head
        qy = yall[:, :qc].reshape(tokens, q_heads, head_dim)
        ky = yall[:, qc:].reshape(tokens, k_heads, head_dim)
        return qy, ky
    qy, _, _ = reference(q_rows, qw, None, eps, dt, weight_bias=weight_bias)
    ky, _, _ = reference(k_rows, kw, None, eps, dt, weight_bias=weight_bias)
    return qy.reshape(tokens, q_heads, head_dim), ky.reshape(tokens, k_heads, head_dim)


# Planted mistakes of the op-by-op cast order.
CAST_MISTAKES = ["cast_single_rounding", "cast_to_f32", "cast_rsqrt_rounded", "cast_weight_before_norm",
                 "cast_trunc", "cast_weight_dropped", "cast_product_ties_away"]


def reference_cast(x, w, residual, eps, dt, mistake=None):
    """The cast order restated: n = RN(h * r), y = RN(n * w) (numpy fp64)."""
    xv = _decode(x, dt)
    e = float(np.float32(eps))
    if residual is not None:
        h = _round(xv + _decode(residual, dt), dt)
        h_store = _encode(h, dt)
    else:
        h = xv
        h_store = None
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        r = 1.0 / np.sqrt((h * h).sum(axis=1, keepdims=True) / h.shape[1] + e)
        wv = None if (w is None or mistake == "cast_weight_dropped") else _decode(w, dt)
        if mistake == "cast_rsqrt_rounded":
            r = _round(r, dt)
        v = h * r
        if mistake == "cast_single_rounding":
            y = v if wv is None else v * wv
        elif mistake == "cast_weight_before_norm":
            y = _round(h * wv, dt) * r if wv is not None else v
        else:
            n = _round(v, "f32" if mistake == "cast_to_f32" else dt, "trunc" if mistake == "cast_trunc" else "rne")
            y = n if wv is None else n * wv
    return _encode(_round(y, dt, "away" if mistake == "cast_product_ties_away" else "rne"), dt), h_store, v


LN_MISTAKES = ["bessel", "eps_outside_sqrt", "no_centering", "bias_inside_weight", "no_bias",
               "stats_from_x", "unrounded_residual", "mean_over_h_minus_1"]


def reference_ln(x, w, b, residual, eps, dt, mistake=None):
    """Independent numpy fp64 LayerNorm with optional planted mistakes."""
    xv = _decode(x, dt)
    e = float(np.float32(eps))
    if residual is not None:
        sm = xv + _decode(residual, dt)
        h_store = _round(sm, dt)
        h = sm if mistake == "unrounded_residual" else h_store
    else:
        h, h_store = xv, None
    st = xv if mistake == "stats_from_x" else h
    n = h.shape[1]
    with np.errstate(invalid="ignore", divide="ignore"):
        mean = st.sum(axis=1, keepdims=True) / (n - 1 if mistake == "mean_over_h_minus_1" else n)
        if mistake == "no_centering":
            mean = np.zeros_like(mean)
        var = ((st - mean) ** 2).sum(axis=1, keepdims=True) / (n - 1 if mistake == "bessel" else n)
        if mistake == "eps_outside_sqrt":
            nrm = (h - mean) / (np.sqrt(var) + e)
        else:
            nrm = (h - mean) / np.sqrt(var + e)
        y = nrm
        if w is not None:
            wv = _decode(w, dt)
            if b is not None and mistake not in ("no_bias",):
                bv = _decode(b, dt)
                y = wv * (nrm + bv) if mistake == "bias_inside_weight" else wv * nrm + bv
            else:
                y = wv * nrm
    out = _encode(_round(y, dt), dt)
    return out, (None if h_store is None else _encode(h_store, dt)), nrm, y


MX_MISTAKES = ["scale_without_offset", "scale_ceil", "no_saturation", "blocks_of_16", "truncate_codes",
               "ties_away_codes", "scale_off_by_one"]


def _e4m3(v, mode="rne", saturate=True):
    """Numpy E4M3 encoder (values -> codes) with a selectable rounding rule."""
    v = np.asarray(v, dtype=np.float64)
    sign = np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    a = np.abs(v)
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        _, e = np.frexp(np.where(a > 0, a, 1.0))
        q = np.maximum(e - 4, -9)
        s = np.ldexp(a, -q)
        n = np.rint(s) if mode == "rne" else np.floor(s) if mode == "trunc" else np.floor(s + 0.5)
        r = np.ldexp(n, q)
    over = r > 448.0
    r = np.where(over, 448.0, r)
    codes = np.zeros(v.shape, dtype=np.uint8)
    sub = r < 2.0 ** -6
    codes = np.where(sub, np.ldexp(r, 9).astype(np.int64), 0)
    _, re_ = np.frexp(np.where(r > 0, r, 1.0))
    f = np.ldexp(r, -(re_ - 1)) - 1.0
    norm = ((re_ - 1 + 7) << 3) | np.rint(f * 8).astype(np.int64)
    codes = np.where(sub, codes, norm).astype(np.uint8)
    if not saturate:
        codes = np.where(over, 0x7F, codes).astype(np.uint8)
    return (codes | sign).astype(np.uint8)


def reference_mx(x, w, residual, eps, dt, weight_bias=0.0, mistake=None):
    """Numpy MXFP8 RMSNorm on top of ``reference`` (fp64 values), with planted mistakes."""
    _, h_out, v = reference(x, w, residual, eps, dt, weight_bias=weight_bias)
    rows, hidden = v.shape
    blk = 16 if mistake == "blocks_of_16" else 32
    vb = v.reshape(rows, hidden // blk, blk)
    amax = np.abs(vb).max(axis=2)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(amax > 0, amax, 1.0))
    e = np.ceil(lg) if mistake == "scale_ceil" else np.floor(lg)
    off = 0 if mistake == "scale_without_offset" else 8
    s = np.where(amax > 0, e - off, -127)
    if mistake == "scale_off_by_one":
        s = s + 1
    s = np.clip(s, -127, 127).astype(np.int64)
    scaled = vb * np.ldexp(1.0, -s)[:, :, None]
    mode = {"truncate_codes": "trunc", "ties_away_codes": "away"}.get(mistake, "rne")
    codes = _e4m3(scaled, mode=mode, saturate=mistake != "no_saturation").reshape(rows, hidden)
    scales = (s + 127).astype(np.uint8)
    if blk == 16:
        scales = scales[:, ::2]
    return codes, scales, h_out, v


NV_MISTAKES = ["nv_no_div6", "nv_blocks_of_32", "nv_truncate", "nv_no_saturation", "nv_nibbles_swapped",
               "nv_tensor_scale_ignored", "nv_scale_ceil"]


def _e2m1(v, mode="rne", saturate=True):
    a = np.abs(np.asarray(v, dtype=np.float64))
    sign = np.where(np.signbit(v), 0x8, 0)
    q = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    s = a / q
    n = np.rint(s) if mode == "rne" else np.floor(s) if mode == "trunc" else np.ceil(s)
    r = n * q
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    if saturate:
        r = np.minimum(r, 6.0)
        idx = np.searchsorted(mags, r)
    else:
        idx = np.where(r > 6.0, 0, np.searchsorted(mags, np.minimum(r, 6.0)))   # overflow wraps to 0
    return (sign | idx).astype(np.uint8)


def reference_nv(x, w, residual, eps, dt, weight_bias=0.0, tensor_scale=1.0, mistake=None):
    """Numpy NVFP4 RMSNorm on top of ``reference`` with planted mistakes."""
    _, h_out, v = reference(x, w, residual, eps, dt, weight_bias=weight_bias)
    rows, hidden = v.shape
    blk = 32 if mistake == "nv_blocks_of_32" else 16
    S = 1.0 if mistake == "nv_tensor_scale_ignored" else float(np.float32(tensor_scale))
    vb = v.reshape(rows, hidden // blk, blk)
    amax = np.abs(vb).max(axis=2)
    div = 1.0 if mistake == "nv_no_div6" else 6.0
    t = amax / (div * S)
    sc = _e4m3(t) if mistake != "nv_scale_ceil" else _e4m3(t * (1 + 2 ** -4))
    sv = np.where((sc & 0x7F) == 0, 0.0, _e4m3_values_np(sc))
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(sv[:, :, None] > 0, vb / (sv[:, :, None] * S), 0.0)
    mode = "trunc" if mistake == "nv_truncate" else "rne"
    codes = _e2m1(scaled, mode=mode, saturate=mistake != "nv_no_saturation").reshape(rows, hidden)
    lo, hi = codes[:, 0::2], codes[:, 1::2]
    packed = (hi | (lo << 4)) if mistake == "nv_nibbles_swapped" else (lo | (hi << 4))
    scales = sc if blk == 16 else np.repeat(sc, 2, axis=1)
    return packed.astype(np.uint8), scales.astype(np.uint8), h_out, v


def _e4m3_values_np(codes):
    c = np.asarray(codes, dtype=np.int64)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    return np.where(ef == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * np.ldexp(1.0, ef - 7))
