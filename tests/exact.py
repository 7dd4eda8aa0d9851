"""Exact rational arithmetic used to pin the oracle (brute force on tiny rows).

Nothing here shares code with the oracle or the CUDA library.  Floating-point
formats are decoded from their IEEE definitions into ``fractions.Fraction``,
and a result of the form ``sign * sqrt(q)`` with ``q`` rational is rounded to
the nearest representable value (ties to even) by comparing ``q`` with exact
squares of the candidate values and of the midpoints between them.  No
floating-point operation takes part in a decision.
"""
from __future__ import annotations

from fractions import Fraction

# (exponent bits, fraction bits) of the formats the path uses.
FORMATS = {"bf16": (8, 7), "f32": (8, 23)}


def _fmt(fmt):
    e_bits, f_bits = FORMATS[fmt]
    bias = (1 << (e_bits - 1)) - 1
    inf_ord = ((1 << e_bits) - 1) << f_bits        # ordinal of +inf
    return e_bits, f_bits, bias, inf_ord


def decode(bits: int, fmt: str):
    """Exact value of a finite encoding as a Fraction (None for inf/NaN)."""
    e_bits, f_bits, bias, _ = _fmt(fmt)
    sign = -1 if (bits >> (e_bits + f_bits)) & 1 else 1
    e = (bits >> f_bits) & ((1 << e_bits) - 1)
    f = bits & ((1 << f_bits) - 1)
    if e == (1 << e_bits) - 1:
        return None
    if e == 0:
        mag = Fraction(f, 1 << f_bits) * Fraction(2) ** (1 - bias)
    else:
        mag = (1 + Fraction(f, 1 << f_bits)) * Fraction(2) ** (e - bias)
    return sign * mag


def _ord_value(k: int, fmt: str) -> Fraction:
    """Value of positive ordinal k; the +inf ordinal stands for 2^(emax+1)."""
    e_bits, f_bits, bias, inf_ord = _fmt(fmt)
    if k == inf_ord:
        return Fraction(2) ** (bias + 1)
    return decode(k, fmt)


def round_sqrt(sign: int, q: Fraction, fmt: str) -> int:
    """Bits of the correctly rounded (nearest, ties to even) value sign*sqrt(q), q >= 0."""
    e_bits, f_bits, bias, inf_ord = _fmt(fmt)
    sign_bit = (1 << (e_bits + f_bits)) if sign < 0 else 0
    if q == 0:
        return sign_bit
    # largest ordinal k with value(k)^2 <= q (k may be the inf ordinal's predecessor)
    lo, hi = 0, inf_ord
    if _ord_value(inf_ord, fmt) ** 2 <= q:
        return sign_bit | inf_ord
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _ord_value(mid, fmt) ** 2 <= q:
            lo = mid
        else:
            hi = mid
    a, b = _ord_value(lo, fmt), _ord_value(hi, fmt)
    m2 = ((a + b) / 2) ** 2
    if q < m2:
        k = lo
    elif q > m2:
        k = hi
    else:
        k = lo if lo % 2 == 0 else hi
    return sign_bit | k


def round_value(v: Fraction, fmt: str) -> int:
    """Bits of the correctly rounded value of a rational v."""
    return round_sqrt(-1 if v < 0 else 1, v * v, fmt)


def midpoint_distance(sign_q: Fraction, fmt: str) -> Fraction:
    """Relative distance |q - m^2| / m^2 from q to the nearest rounding midpoint squared."""
    q = sign_q
    e_bits, f_bits, bias, inf_ord = _fmt(fmt)
    lo, hi = 0, inf_ord
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _ord_value(mid, fmt) ** 2 <= q:
            lo = mid
        else:
            hi = mid
    best = None
    for k in (lo - 1, lo, hi):
        if k < 0 or k + 1 > inf_ord:
            continue
        m2 = ((_ord_value(k, fmt) + _ord_value(k + 1, fmt)) / 2) ** 2
        d = abs(q - m2) / m2
        best = d if best is None else min(best, d)
    return best


def rmsnorm_row_exact(x, w, residual, eps_bits_value: Fraction, fmt: str, weight_bias: Fraction = Fraction(0)):
    """Exact RMSNorm of one row given as lists of encodings (ints).

    The weight enters as (w_i + weight_bias).  Returns (y_bits,
    residual_out_bits or None, q_list, signs) where y_i = sign_i * sqrt(q_i)
    exactly, before rounding.
    """
    n = len(x)
    xs = [decode(b, fmt) for b in x]
    if residual is not None:
        rs = [decode(b, fmt) for b in residual]
        h_bits = [round_value(a + b, fmt) for a, b in zip(xs, rs)]
        hs = [decode(b, fmt) for b in h_bits]
    else:
        h_bits = None
        hs = xs
    ws = [decode(b, fmt) + weight_bias for b in w] if w is not None else [Fraction(1)] * n
    s = sum(h * h for h in hs)
    denom = s / n + eps_bits_value
    qs, signs, y_bits = [], [], []
    sign_mask = 1 << (sum(FORMATS[fmt]))
    for i in range(n):
        p = hs[i] * ws[i]
        q = p * p / denom
        if p != 0:
            sg = -1 if p < 0 else 1
        else:
            # IEEE sign of a zero product: XOR of the operand signs (r > 0)
            hb = (h_bits[i] if h_bits is not None else x[i]) & sign_mask
            if w is None:
                wneg = False
            elif ws[i] != 0:
                wneg = ws[i] < 0
            elif weight_bias == 0:
                wneg = (w[i] & sign_mask) != 0
            else:
                wneg = False   # w + b == 0 exactly: IEEE round-to-nearest sum is +0
            sg = -1 if (hb != 0) != wneg else 1
        qs.append(q)
        signs.append(sg)
        y_bits.append(round_sqrt(sg, q, fmt))
    return y_bits, h_bits, qs, signs


def rmsnorm_cast_row_exact(x, w, residual, eps_bits_value: Fraction, fmt: str):
    """Exact RMSNorm of one row in the op-by-op cast order: the normalised
    value is rounded to the format, then multiplied by the weight and rounded
    again.  Returns (y_bits, residual_out_bits or None, n_bits, q_list, signs),
    where n_bits are the rounded normalised values and sign_i * sqrt(q_i) their
    exact values."""
    n_bits, h_bits, qs, signs = rmsnorm_row_exact(x, None, residual, eps_bits_value, fmt)
    if w is None:
        return list(n_bits), h_bits, n_bits, qs, signs
    return [cast_times_weight(nb, wb, fmt) for nb, wb in zip(n_bits, w)], h_bits, n_bits, qs, signs


def cast_times_weight(n_bits: int, w_bits: int, fmt: str) -> int:
    """Bits of RN(n * w) for two encodings (IEEE sign of an exact zero product)."""
    sign_mask = 1 << (sum(FORMATS[fmt]))
    p = decode(n_bits, fmt) * decode(w_bits, fmt)
    if p == 0:
        return sign_mask if ((n_bits & sign_mask) != 0) != ((w_bits & sign_mask) != 0) else 0
    return round_value(p, fmt)


def neighbours(bits: int, fmt: str):
    """The encodings adjacent to a finite nonzero encoding of the same sign."""
    sign_mask = 1 << (sum(FORMATS[fmt]))
    mag = bits & (sign_mask - 1)
    out = []
    for m in (mag - 1, mag + 1):
        if m >= 0:
            out.append((bits & sign_mask) | m)
    return out


def _cmp_affine_sqrt(a: Fraction, d: Fraction, b: Fraction, v: Fraction) -> int:
    """Sign of (a / sqrt(d) + b) - v, exactly (d > 0)."""
    c = v - b                      # compare a / sqrt(d) with c
    if a >= 0 and c <= 0:
        return 0 if (a == 0 and c == 0) else 1
    if a <= 0 and c >= 0:
        return -1
    lhs, rhs = a * a, c * c * d    # same signs: compare squares
    if a > 0:
        return (lhs > rhs) - (lhs < rhs)
    return (rhs > lhs) - (rhs < lhs)


def round_affine_sqrt(a: Fraction, d: Fraction, b: Fraction, fmt: str) -> int:
    """Bits of the correctly rounded value of a / sqrt(d) + b (d > 0), ties to even."""
    e_bits, f_bits, bias, inf_ord = _fmt(fmt)
    sign_bit = 1 << (e_bits + f_bits)
    s0 = _cmp_affine_sqrt(a, d, b, Fraction(0))
    if s0 == 0:
        return 0
    neg = s0 < 0
    if neg:                        # round the magnitude of -(value)
        a, b = -a, -b
    # largest ordinal k with value(k) <= value (positive side)
    lo, hi = 0, inf_ord
    if _cmp_affine_sqrt(a, d, b, _ord_value(inf_ord, fmt)) >= 0:
        return (sign_bit if neg else 0) | inf_ord
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _cmp_affine_sqrt(a, d, b, _ord_value(mid, fmt)) >= 0:
            lo = mid
        else:
            hi = mid
    m = (_ord_value(lo, fmt) + _ord_value(hi, fmt)) / 2
    c = _cmp_affine_sqrt(a, d, b, m)
    k = lo if c < 0 else hi if c > 0 else (lo if lo % 2 == 0 else hi)
    return (sign_bit if neg else 0) | k


def near_midpoint_affine(a: Fraction, d: Fraction, b: Fraction, bits1: int, bits2: int, fmt: str,
                         rel: Fraction = Fraction(1, 2 ** 44)) -> bool:
    """True if a / sqrt(d) + b lies within `rel` (relative) of the midpoint of
    two adjacent encodings bits1, bits2 (an fp64 computation may round it either way)."""
    v1, v2 = decode(bits1, fmt), decode(bits2, fmt)
    if v1 is None or v2 is None:
        return False
    m = (v1 + v2) / 2
    lo, hi = m - abs(m) * rel, m + abs(m) * rel
    return _cmp_affine_sqrt(a, d, b, lo) >= 0 and _cmp_affine_sqrt(a, d, b, hi) <= 0


def layernorm_row_exact(x, w, b, residual, eps_value: Fraction, fmt: str, want_terms: bool = False):
    """Exact LayerNorm of one row of encodings: y_i = w_i (h_i - mean) / sqrt(var + eps) + b_i,
    correctly rounded.  Returns (y_bits, residual_out_bits or None), plus the
    exact terms (a_i, d, b_i) of y_i = a_i / sqrt(d) + b_i with ``want_terms``."""
    n = len(x)
    xs = [decode(v, fmt) for v in x]
    if residual is not None:
        rs = [decode(v, fmt) for v in residual]
        h_bits = [round_value(p + q, fmt) for p, q in zip(xs, rs)]
        hs = [decode(v, fmt) for v in h_bits]
    else:
        h_bits, hs = None, xs
    mean = sum(hs) / n
    var = sum((h - mean) ** 2 for h in hs) / n
    d = var + eps_value
    ws = [decode(v, fmt) for v in w] if w is not None else [Fraction(1)] * n
    bs = [decode(v, fmt) for v in b] if b is not None else [Fraction(0)] * n
    out = []
    terms = []
    for i in range(n):
        out.append(round_affine_sqrt(ws[i] * (hs[i] - mean), d, bs[i], fmt))
        terms.append((ws[i] * (hs[i] - mean), d, bs[i]))
    if want_terms:
        return out, h_bits, terms
    return out, h_bits



# ---------------------------------------------------------------- E4M3, MXFP8
# FP8 E4M3 (OCP): 4 exponent bits (bias 7), 3 fraction bits, no infinities,
# S.1111.111 is NaN, largest finite 448, subnormal quantum 2^-9.

def e4m3_decode(code: int):
    """Exact value of an E4M3 code (None for NaN)."""
    sign = -1 if code & 0x80 else 1
    ef = (code >> 3) & 0xF
    m = code & 0x7
    if ef == 0xF and m == 0x7:
        return None
    if ef == 0:
        return sign * Fraction(m, 8) * Fraction(1, 64)
    return sign * (1 + Fraction(m, 8)) * Fraction(2) ** (ef - 7)


def e4m3_round_sqrt_sat(sign: int, q: Fraction) -> int:
    """E4M3 code of sign*sqrt(q): nearest, ties to even, magnitudes above 448 -> 448."""
    sign_bit = 0x80 if sign < 0 else 0
    if q == 0:
        return sign_bit
    if q >= 448 * 448:
        return sign_bit | 0x7E
    lo, hi = 0, 0x7E          # positive codes are ordered by value
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if e4m3_decode(mid) ** 2 <= q:
            lo = mid
        else:
            hi = mid
    if e4m3_decode(hi) ** 2 <= q:
        lo = hi
    if lo == 0x7E:
        return sign_bit | 0x7E
    a, b = e4m3_decode(lo), e4m3_decode(lo + 1)
    m2 = ((a + b) / 2) ** 2
    k = lo if q < m2 else lo + 1 if q > m2 else (lo if lo % 2 == 0 else lo + 1)
    return sign_bit | k


def floor_log2_sqrt(q: Fraction) -> int:
    """floor(log2(sqrt(q))) for q > 0, exactly."""
    e = 0
    while Fraction(4) ** e > q:
        e -= 1
    while Fraction(4) ** (e + 1) <= q:
        e += 1
    return e


def mxfp8_row_exact(x, w, residual, eps_value: Fraction, fmt: str, weight_bias: Fraction = Fraction(0)):
    """Exact MXFP8 codes and E8M0 scales of one row (hidden a multiple of 32)."""
    n = len(x)
    xs = [decode(b, fmt) for b in x]
    if residual is not None:
        rs = [decode(b, fmt) for b in residual]
        hs = [decode(round_value(a + b, fmt), fmt) for a, b in zip(xs, rs)]
    else:
        hs = xs
    ws = [decode(b, fmt) + weight_bias for b in w] if w is not None else [Fraction(1)] * n
    denom = sum(h * h for h in hs) / n + eps_value
    codes, scales, qs = [], [], []
    for k in range(n // 32):
        ps = [hs[i] * ws[i] for i in range(32 * k, 32 * k + 32)]
        q_block = [p * p / denom for p in ps]        # v_i^2
        amax2 = max(q_block)
        s = -127 if amax2 == 0 else max(-127, min(127, floor_log2_sqrt(amax2) - 8))
        scales.append(s + 127)
        for p, q in zip(ps, q_block):
            codes.append(e4m3_round_sqrt_sat(-1 if p < 0 else 1, q * Fraction(4) ** (-s)))
            qs.append(q * Fraction(4) ** (-s))
    return codes, scales, qs



# ---------------------------------------------------------------- E2M1, NVFP4
E2M1_MAGS = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4),
             Fraction(6)]


def e2m1_decode(code: int) -> Fraction:
    return (-1 if code & 0x8 else 1) * E2M1_MAGS[code & 0x7]


def e2m1_round_sqrt_sat(sign: int, q: Fraction) -> int:
    """E2M1 code of sign*sqrt(q): nearest, ties to the even code, saturated at 6."""
    sign_bit = 0x8 if sign < 0 else 0
    if q >= 36:
        return sign_bit | 7
    lo = max(i for i in range(8) if E2M1_MAGS[i] ** 2 <= q)
    if lo == 7:
        return sign_bit | 7
    m2 = ((E2M1_MAGS[lo] + E2M1_MAGS[lo + 1]) / 2) ** 2
    k = lo if q < m2 else lo + 1 if q > m2 else (lo if lo % 2 == 0 else lo + 1)
    return sign_bit | k


def nvfp4_row_exact(x, w, residual, eps_value: Fraction, fmt: str, tensor_scale: Fraction,
                    weight_bias: Fraction = Fraction(0)):
    """Exact NVFP4 codes (4-bit, unpacked) and E4M3 block scales of one row
    (hidden a multiple of 16), with the reading: scale = E4M3(amax / (6 S)),
    code = E2M1(v / (scale S)).  Returns (codes, scales, q_code_list)."""
    n = len(x)
    xs = [decode(b, fmt) for b in x]
    if residual is not None:
        rs = [decode(b, fmt) for b in residual]
        hs = [decode(round_value(a + b, fmt), fmt) for a, b in zip(xs, rs)]
    else:
        hs = xs
    ws = [decode(b, fmt) + weight_bias for b in w] if w is not None else [Fraction(1)] * n
    denom = sum(h * h for h in hs) / n + eps_value
    codes, scales, qs = [], [], []
    for k in range(n // 16):
        ps = [hs[i] * ws[i] for i in range(16 * k, 16 * k + 16)]
        q_block = [p * p / denom for p in ps]                   # v_i^2
        sc = e4m3_round_sqrt_sat(1, max(q_block) / (6 * tensor_scale) ** 2)
        scales.append(sc)
        sv = e4m3_decode(sc)
        for p, q in zip(ps, q_block):
            if sv == 0:
                codes.append(0)
                qs.append(Fraction(0))
            else:
                qq = q / (sv * tensor_scale) ** 2
                codes.append(e2m1_round_sqrt_sat(-1 if p < 0 else 1, qq))
                qs.append(qq)
    return codes, scales, qs
