"""Pins for an RMSNorm reference implementation: facts fixed by the definition
and by mathematics, not by any implementation.

Each ``pin_*`` takes ``impl(x, w, residual, eps, dtype) -> (y, residual_out, y_exact)``
with numpy arrays in the oracle's convention (bf16 as uint16 bits, fp32 as
float32) and returns a list of failure messages (empty when the pin holds).
The same pins run against the oracle (all must hold) and against deliberately
broken variants of it (each must be caught by at least one pin).

Where the definition comes from: "Building a GPU compiler from scratch: from
PyTorch to CUDA via multi-level IR (Emmy)" -- running example and section
"Tensor IR".  Expected values are derived with exact rational arithmetic
(``tests/exact.py``) or are closed forms / invariants of that definition.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

import exact

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.txt")
SIGN_MASK = {"bf16": 0x8000, "f32": 0x80000000}


# ---------------------------------------------------------------- helpers

def bits_of(a, dtype):
    a = np.ascontiguousarray(a)
    return a.astype(np.uint16) if dtype == "bf16" else a.view(np.uint32)


def encode_exact(v: Fraction, dtype):
    """Encoding of an exactly representable rational (raises if not exact)."""
    b = exact.round_value(v, dtype)
    if exact.decode(b, dtype) != v:
        raise ValueError(f"{v} is not representable in {dtype}")
    if v == 0:
        b = 0
    return b


def to_array(bits_list, dtype):
    if dtype == "bf16":
        return np.array(bits_list, dtype=np.uint16)
    return np.array(bits_list, dtype=np.uint32).view(np.float32)


def f32_exact(eps) -> Fraction:
    return Fraction(float(np.float32(eps)))


def _expand(tokens):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.split("*")
            out.extend([v] * int(n))
        else:
            out.append(t)
    return out


def parse_golden(path=GOLDEN):
    cases, cur = [], None
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "case":
            cur = {"name": rest[0]}
            cases.append(cur)
            continue
        if key == "dtype":
            cur["dtype"] = rest[0]
        elif key == "eps":
            cur["eps"] = Fraction(rest[0])
        elif key in ("x", "w", "residual", "y2", "resout"):
            cur[key] = None if rest == ["-"] else [Fraction(t) for t in _expand(rest)]
        elif key == "sign":
            cur["sign"] = [-1 if t == "-" else 1 for t in _expand(rest)]
        else:
            raise ValueError(f"unknown key {key!r} in {path}")
    return cases


def random_bits(rng, dtype, n, lo_exp=-6, hi_exp=6):
    """Random finite encodings: random sign and fraction, exponent in a range
    that keeps squares and sums far from overflow and underflow."""
    if dtype == "bf16":
        e_bits, f_bits, bias = 8, 7, 127
    else:
        e_bits, f_bits, bias = 8, 23, 127
    sign = rng.integers(0, 2, n)
    e = rng.integers(lo_exp + bias, hi_exp + bias + 1, n)
    f = rng.integers(0, 1 << f_bits, n)
    bits = (sign << (e_bits + f_bits)) | (e << f_bits) | f
    return [int(b) for b in bits]


# ---------------------------------------------------------------- pins

def pin_golden(impl):
    """Hand-derived closed-form cases stored in tests/golden/closed_forms.txt."""
    fails = []
    for c in parse_golden():
        dt = c["dtype"]
        n = len(c["x"])
        x = to_array([encode_exact(v, dt) for v in c["x"]], dt).reshape(1, n)
        w = None if c["w"] is None else to_array([encode_exact(v, dt) for v in c["w"]], dt)
        res = None if c["residual"] is None else to_array(
            [encode_exact(v, dt) for v in c["residual"]], dt).reshape(1, n)
        eps = float(c["eps"])
        y, rout, _ = impl(x, w, res, eps, dt)
        want = [exact.round_sqrt(s, q, dt) for s, q in zip(c["sign"], c["y2"])]
        got = [int(b) for b in bits_of(y, dt).reshape(-1)]
        if got != want:
            fails.append(f"golden {c['name']}: y bits {got[:8]} != {want[:8]}")
        if c.get("resout") is not None:
            want_r = [encode_exact(v, dt) for v in c["resout"]]
            got_r = [int(b) for b in bits_of(rout, dt).reshape(-1)] if rout is not None else None
            if got_r != want_r:
                fails.append(f"golden {c['name']}: residual_out {got_r} != {want_r}")
    return fails


def pin_bruteforce(impl, n_cases=60, seed=1234):
    """Random tiny rows (hidden 1..8, three rows each), every option combination,
    checked bit for bit against the exactly rounded rational answer."""
    rng = np.random.default_rng(seed)
    fails = []
    eps_choices = [0.0, 1e-6, 1e-5, 0.25, 3.0]
    for k in range(n_cases):
        dt = ("bf16", "f32")[k % 2]
        has_w = bool((k // 2) % 2)
        has_res = bool((k // 4) % 2)
        hidden = int(rng.integers(1, 9))
        rows = 3
        eps = eps_choices[k % len(eps_choices)]
        xb = [random_bits(rng, dt, hidden) for _ in range(rows)]
        rb = [random_bits(rng, dt, hidden) for _ in range(rows)] if has_res else None
        wb = random_bits(rng, dt, hidden, -2, 2) if has_w else None
        x = to_array(sum(xb, []), dt).reshape(rows, hidden)
        res = to_array(sum(rb, []), dt).reshape(rows, hidden) if has_res else None
        w = to_array(wb, dt) if has_w else None
        y, rout, _ = impl(x, w, res, eps, dt)
        yb = bits_of(y, dt).reshape(rows, hidden)
        for r in range(rows):
            want, want_h, qs, signs = exact.rmsnorm_row_exact(
                xb[r], wb, rb[r] if has_res else None, f32_exact(eps), dt)
            for i in range(hidden):
                if int(yb[r, i]) != want[i]:
                    d = exact.midpoint_distance(qs[i], dt)
                    if d is None or d > Fraction(1, 2 ** 44):
                        fails.append(f"bruteforce case {k} ({dt}, w={has_w}, res={has_res}, "
                                     f"H={hidden}, eps={eps}) row {r} elem {i}: "
                                     f"{int(yb[r, i]):#x} != {want[i]:#x}")
            if has_res:
                got_h = [int(b) for b in bits_of(rout, dt).reshape(rows, hidden)[r]]
                if got_h != want_h:
                    fails.append(f"bruteforce case {k}: residual_out row {r} {got_h} != {want_h}")
    return fails


def pin_constant_row(impl):
    """x_i = c for every i: y_i = c / sqrt(c^2 + eps) * w_i (closed form)."""
    fails = []
    rng = np.random.default_rng(7)
    for dt in ("bf16", "f32"):
        for hidden in (1, 7, 576, 4096):
            for c in (Fraction(3, 4), Fraction(-5, 2), Fraction(1, 64)):
                for eps in (0.0, 1e-5, 0.5):
                    cb = encode_exact(c, dt)
                    x = to_array([cb] * hidden, dt).reshape(1, hidden)
                    wb = random_bits(rng, dt, hidden, -1, 1)
                    w = to_array(wb, dt)
                    y, _, _ = impl(x, w, None, eps, dt)
                    e = f32_exact(eps)
                    got = bits_of(y, dt).reshape(-1)
                    for i in (0, hidden // 2, hidden - 1):
                        wi = exact.decode(wb[i], dt)
                        p = c * wi
                        q = p * p / (c * c + e)
                        want = exact.round_sqrt(-1 if p < 0 else 1, q, dt)
                        if int(got[i]) != want:
                            fails.append(f"constant row {dt} H={hidden} c={c} eps={eps} i={i}: "
                                         f"{int(got[i]):#x} != {want:#x}")
    return fails


def pin_scale_invariance(impl):
    """With eps = 0, y(a*x) = sign(a) * y(x) for a power of two a (bit-exact in
    the I/O type, since the scaled inputs are exact); also y(-x) = -y(x)."""
    fails = []
    rng = np.random.default_rng(11)
    for dt in ("bf16", "f32"):
        for hidden in (5, 64, 1000):
            xb = random_bits(rng, dt, 4 * hidden, -3, 3)
            x = to_array(xb, dt).reshape(4, hidden)
            w = to_array(random_bits(rng, dt, hidden, -1, 1), dt)
            y0, _, y0e = impl(x, w, None, 0.0, dt)
            for a in (2.0 ** 5, 2.0 ** -7, -1.0, -(2.0 ** 3)):
                if dt == "bf16":
                    xf = np.array(xb, dtype=np.uint32) << 16
                    xs = (xf.view(np.float32) * np.float32(a)).view(np.uint32) >> 16
                    xa = xs.astype(np.uint16).reshape(4, hidden)
                else:
                    xa = (x * np.float32(a)).astype(np.float32)
                ya, _, _ = impl(xa, w, None, 0.0, dt)
                b0 = bits_of(y0, dt).astype(np.uint64)
                ba = bits_of(ya, dt).astype(np.uint64)
                if a < 0:
                    b0 = b0 ^ SIGN_MASK[dt]
                if not np.array_equal(b0, ba):
                    fails.append(f"scale invariance {dt} H={hidden} a={a}: "
                                 f"{int((b0 != ba).sum())} elements differ")
    return fails


def pin_unit_rms(impl):
    """With no weight and eps = 0, the fp64 result has mean(y^2) = 1."""
    fails = []
    rng = np.random.default_rng(5)
    for dt in ("bf16", "f32"):
        for hidden in (3, 128, 2048):
            x = to_array(random_bits(rng, dt, 5 * hidden, -4, 4), dt).reshape(5, hidden)
            _, _, ye = impl(x, None, None, 0.0, dt)
            if ye is None:
                fails.append("unit rms: no fp64 result")
                continue
            m = (ye * ye).mean(axis=1)
            if not np.all(np.abs(m - 1.0) < 1e-12):
                fails.append(f"unit rms {dt} H={hidden}: mean(y^2) = {m}")
    return fails


def pin_special_values(impl):
    """NaN, infinity and zero rows follow IEEE arithmetic of the definition."""
    fails = []
    for dt in ("bf16", "f32"):
        one = encode_exact(Fraction(1), dt)
        two = encode_exact(Fraction(2), dt)
        nan = 0x7FC0 if dt == "bf16" else 0x7FC00000
        inf = 0x7F80 if dt == "bf16" else 0x7F800000
        x = to_array([one, two, nan, one,    # NaN row -> all NaN
                      one, inf, two, 0,      # inf row -> inf*0 = NaN at inf, 0 elsewhere
                      0, 0, 0, 0], dt).reshape(3, 4)  # zero row, eps > 0 -> zeros
        y, _, _ = impl(x, None, None, 1e-5, dt)
        yv = (np.array(bits_of(y, dt), dtype=np.uint32) << 16).view(np.float32) if dt == "bf16" \
            else np.asarray(y, dtype=np.float32)
        yv = yv.reshape(3, 4)
        if not np.all(np.isnan(yv[0])):
            fails.append(f"special {dt}: NaN row gave {yv[0]}")
        if not (np.isnan(yv[1, 1]) and np.all(yv[1, [0, 2, 3]] == 0)):
            fails.append(f"special {dt}: inf row gave {yv[1]}")
        if not np.all(yv[2] == 0):
            fails.append(f"special {dt}: zero row gave {yv[2]}")
        # eps = 0 on a zero row: 0 * (1 / sqrt(0)) = 0 * inf = NaN
        y0, _, _ = impl(to_array([0, 0], dt).reshape(1, 2), None, None, 0.0, dt)
        y0v = (np.array(bits_of(y0, dt), dtype=np.uint32) << 16).view(np.float32) if dt == "bf16" \
            else np.asarray(y0, dtype=np.float32)
        if not np.all(np.isnan(y0v)):
            fails.append(f"special {dt}: zero row with eps=0 gave {y0v}")
    return fails


def pin_single_element(impl):
    """hidden = 1: y = x * w / sqrt(x^2 + eps)."""
    fails = []
    rng = np.random.default_rng(3)
    for dt in ("bf16", "f32"):
        xb = random_bits(rng, dt, 16, -3, 3)
        wb = random_bits(rng, dt, 1, -1, 1)
        x = to_array(xb, dt).reshape(16, 1)
        w = to_array(wb, dt)
        for eps in (0.0, 1e-6, 2.0):
            y, _, _ = impl(x, w, None, eps, dt)
            got = bits_of(y, dt).reshape(-1)
            e = f32_exact(eps)
            wv = exact.decode(wb[0], dt)
            for i, b in enumerate(xb):
                xv = exact.decode(b, dt)
                p = xv * wv
                want = exact.round_sqrt(-1 if p < 0 else 1, p * p / (xv * xv + e), dt)
                if int(got[i]) != want:
                    fails.append(f"single element {dt} eps={eps}: {int(got[i]):#x} != {want:#x}")
    return fails


def pin_row_independence(impl):
    """Each row is normalised on its own: a batch equals its rows run one by one."""
    fails = []
    rng = np.random.default_rng(9)
    for dt in ("bf16", "f32"):
        x = to_array(random_bits(rng, dt, 6 * 33, -5, 5), dt).reshape(6, 33)
        r = to_array(random_bits(rng, dt, 6 * 33, -5, 5), dt).reshape(6, 33)
        w = to_array(random_bits(rng, dt, 33, -1, 1), dt)
        yb, hb, _ = impl(x, w, r, 1e-6, dt)
        for i in range(6):
            yi, hi, _ = impl(x[i:i + 1], w, r[i:i + 1], 1e-6, dt)
            if not (np.array_equal(bits_of(yi, dt), bits_of(yb[i:i + 1], dt))
                    and np.array_equal(bits_of(hi, dt), bits_of(hb[i:i + 1], dt))):
                fails.append(f"row independence {dt}: row {i} differs")
    return fails


def pin_eps_dominated(impl):
    """Rows far below eps: y_i ~ c * w_i / sqrt(eps), which depends on the exact
    float32 value of eps (the value the caller passes); every element is checked."""
    fails = []
    rng = np.random.default_rng(21)
    for dt in ("bf16", "f32"):
        hidden = 4096
        c = Fraction(1, 2 ** 20)
        x = to_array([encode_exact(c, dt)] * hidden, dt).reshape(1, hidden)
        wb = random_bits(rng, dt, hidden, -1, 1)
        w = to_array(wb, dt)
        for eps in (1e-6, 1e-5):
            y, _, _ = impl(x, w, None, eps, dt)
            got = bits_of(y, dt).reshape(-1)
            e = f32_exact(eps)
            bad = 0
            for i in range(hidden):
                p = c * exact.decode(wb[i], dt)
                want = exact.round_sqrt(-1 if p < 0 else 1, p * p / (c * c + e), dt)
                bad += int(got[i]) != want
            if bad:
                fails.append(f"eps-dominated {dt} eps={eps}: {bad} of {hidden} elements differ")
    return fails


def pin_near_ties(impl, trials=400_000, seed=77):
    """bf16 outputs whose exact value lies within 2^-20 (relative) of a rounding
    midpoint, found by a seeded search over random two-element rows; each is
    checked against the exactly rounded answer.  A result rounded twice (to
    fp32 first, then to bf16) fails here."""
    rng = np.random.default_rng(seed)
    dt = "bf16"
    xb = np.array(random_bits(rng, dt, 2 * trials, -4, 4), dtype=np.uint32).reshape(trials, 2)
    wb = np.array(random_bits(rng, dt, 2, -1, 1), dtype=np.uint32)
    xv = (xb << 16).view(np.float32).astype(np.float64)
    wv = (wb << 16).view(np.float32).astype(np.float64)
    y = xv * wv / np.sqrt((xv * xv).mean(axis=1, keepdims=True))
    a = np.abs(y)
    _, e = np.frexp(a)
    scaled = np.ldexp(a, -(e - 8))            # 8 significant bits before the point
    frac = scaled - np.floor(scaled)
    near = np.abs(frac - 0.5) < 2.0 ** -12    # within 2^-20 relative of a midpoint
    rows_idx = np.unique(np.nonzero(near)[0])[:64]
    fails = []
    if len(rows_idx) < 8:
        return [f"near ties: search found only {len(rows_idx)} rows"]
    x = xb[rows_idx].astype(np.uint16)
    w = wb.astype(np.uint16)
    yo, _, _ = impl(x, w, None, 0.0, dt)
    got = bits_of(yo, dt)
    for k, r in enumerate(rows_idx):
        want, _, qs, _ = exact.rmsnorm_row_exact([int(b) for b in xb[r]], [int(b) for b in wb],
                                                 None, Fraction(0), dt)
        for i in range(2):
            if int(got[k, i]) != want[i]:
                d = exact.midpoint_distance(qs[i], dt)
                if d is None or d > Fraction(1, 2 ** 44):
                    fails.append(f"near ties row {r} elem {i}: {int(got[k, i]):#x} != {want[i]:#x}")
    return fails


def pin_weight_bias(impl_b):
    """y = h * r * (w + b): random tiny rows, b in {1, 1/2, -1/4, 3}, with and
    without a residual, bit-exact against exact rational arithmetic; and
    b = 0 gives the plain weighted op bit for bit."""
    rng = np.random.default_rng(31)
    fails = []
    for k in range(40):
        dt = ("bf16", "f32")[k % 2]
        has_res = bool((k // 2) % 2)
        b = (1.0, 0.5, -0.25, 3.0)[(k // 4) % 4]
        hidden = int(rng.integers(1, 9))
        rows = 3
        eps = (0.0, 1e-6, 0.25)[k % 3]
        xb = [random_bits(rng, dt, hidden) for _ in range(rows)]
        rb = [random_bits(rng, dt, hidden) for _ in range(rows)] if has_res else None
        wb = random_bits(rng, dt, hidden, -2, 2)
        x = to_array(sum(xb, []), dt).reshape(rows, hidden)
        res = to_array(sum(rb, []), dt).reshape(rows, hidden) if has_res else None
        w = to_array(wb, dt)
        y, _, _ = impl_b(x, w, res, eps, dt, b)
        yb = bits_of(y, dt).reshape(rows, hidden)
        for r in range(rows):
            want, _, qs, _ = exact.rmsnorm_row_exact(xb[r], wb, rb[r] if has_res else None, f32_exact(eps),
                                                     dt, Fraction(b))
            for i in range(hidden):
                if int(yb[r, i]) != want[i]:
                    d = exact.midpoint_distance(qs[i], dt)
                    if d is None or d > Fraction(1, 2 ** 44):
                        fails.append(f"weight bias {b} case {k} ({dt}, res={has_res}) row {r} elem {i}: "
                                     f"{int(yb[r, i]):#x} != {want[i]:#x}")
        y0, _, _ = impl_b(x, w, res, eps, dt, 0.0)
        y1, _, _ = impl_b(x, w, res, eps, dt, None)
        if not np.array_equal(bits_of(y0, dt), bits_of(y1, dt)):
            fails.append(f"weight bias 0 differs from the plain weighted op (case {k})")
    return fails


def pin_qk_heads(impl_qk):
    """Packed token rows [q heads | k heads | v heads]: every query head is the
    op on that head with q_w, every key head with k_w, each head on its own
    (exact rational check); a head's result does not depend on the others."""
    rng = np.random.default_rng(41)
    fails = []
    for k, (dt, qh, kh, hd, b) in enumerate([("bf16", 4, 2, 8, 0.0), ("f32", 3, 1, 5, 1.0),
                                              ("bf16", 2, 2, 4, 1.0), ("f32", 1, 3, 8, 0.0)]):
        tokens = 3
        cols = (qh + kh + 1) * hd          # one value head after the keys
        xb = random_bits(rng, dt, tokens * cols, -4, 4)
        x = to_array(xb, dt).reshape(tokens, cols)
        qwb = random_bits(rng, dt, hd, -1, 1)
        kwb = random_bits(rng, dt, hd, -1, 1)
        qy, ky = impl_qk(x, qh, kh, hd, to_array(qwb, dt), to_array(kwb, dt), 1e-6, dt, b)
        qy = bits_of(qy, dt).reshape(tokens, qh, hd)
        ky = bits_of(ky, dt).reshape(tokens, kh, hd)
        for t in range(tokens):
            row = xb[t * cols:(t + 1) * cols]
            for j in range(qh + kh):
                head = row[j * hd:(j + 1) * hd]
                wb = qwb if j < qh else kwb
                want, _, qs, _ = exact.rmsnorm_row_exact(head, wb, None, f32_exact(1e-6), dt, Fraction(b))
                got = qy[t, j] if j < qh else ky[t, j - qh]
                for i in range(hd):
                    if int(got[i]) != want[i]:
                        d = exact.midpoint_distance(qs[i], dt)
                        if d is None or d > Fraction(1, 2 ** 44):
                            fails.append(f"qk case {k} token {t} head {j} elem {i}: "
                                         f"{int(got[i]):#x} != {want[i]:#x}")
    return fails


# ------------------------------------------------------------- LayerNorm pins
# impl_ln(x, w, b, residual, eps, dtype) -> (y, residual_out, n_exact, y_exact)
# Definition: "GPT-2 on the GPU", section "The Whole Model as One Kernel".

def pin_ln_bruteforce(impl_ln, n_cases=80, seed=4321):
    """Random tiny rows, every option, bit-exact against exact rational arithmetic."""
    rng = np.random.default_rng(seed)
    fails = []
    for k in range(n_cases):
        dt = ("bf16", "f32")[k % 2]
        has_w = bool((k // 2) % 2)
        has_b = has_w and bool((k // 4) % 2)
        has_res = bool((k // 8) % 2)
        hidden = int(rng.integers(2, 9))
        eps = (0.0, 1e-5, 0.25)[k % 3]
        rows = 3
        xb = [random_bits(rng, dt, hidden) for _ in range(rows)]
        rb = [random_bits(rng, dt, hidden) for _ in range(rows)] if has_res else None
        wb = random_bits(rng, dt, hidden, -2, 2) if has_w else None
        bb = random_bits(rng, dt, hidden, -2, 2) if has_b else None
        x = to_array(sum(xb, []), dt).reshape(rows, hidden)
        res = to_array(sum(rb, []), dt).reshape(rows, hidden) if has_res else None
        w = to_array(wb, dt) if has_w else None
        b = to_array(bb, dt) if has_b else None
        y, rout, _, _ = impl_ln(x, w, b, res, eps, dt)
        yb = bits_of(y, dt).reshape(rows, hidden)
        for r in range(rows):
            want, want_h, terms = exact.layernorm_row_exact(xb[r], wb, bb, rb[r] if has_res else None,
                                                            f32_exact(eps), dt, want_terms=True)
            got = [int(v) for v in yb[r]]
            for i in range(hidden):
                # a mismatch is allowed only for a value within 2^-44 of a rounding midpoint
                if got[i] != want[i] and not exact.near_midpoint_affine(*terms[i], got[i], want[i], dt):
                    fails.append(f"ln bruteforce case {k} ({dt}, w={has_w}, b={has_b}, res={has_res},"
                                 f" eps={eps}) row {r} elem {i}: {got[i]:#x} != {want[i]:#x}")
            if has_res and [int(v) for v in bits_of(rout, dt).reshape(rows, hidden)[r]] != want_h:
                fails.append(f"ln bruteforce case {k}: residual_out row {r}")
    return fails


def pin_ln_closed_forms(impl_ln):
    """Hand-derived cases: [1, 2, 3, 4] (mean 5/2, variance 5/4: n_i^2 =
    (x_i - 5/2)^2 / (5/4) = 9/5, 1/5, 1/5, 9/5); a constant row gives y = b
    exactly (n = 0, eps > 0); [a, -a] gives n = +-a / sqrt(a^2 + eps)."""
    fails = []
    for dt in ("bf16", "f32"):
        x = to_array([encode_exact(Fraction(v), dt) for v in (1, 2, 3, 4)], dt).reshape(1, 4)
        y, _, _, _ = impl_ln(x, None, None, None, 0.0, dt)
        want = [exact.round_sqrt(s, q, dt) for s, q in zip((-1, -1, 1, 1),
                                                              (Fraction(9, 5), Fraction(1, 5), Fraction(1, 5),
                                                               Fraction(9, 5)))]
        if [int(v) for v in bits_of(y, dt).reshape(-1)] != want:
            fails.append(f"ln [1,2,3,4] {dt}")
        c = encode_exact(Fraction(3, 4), dt)
        bvals = [Fraction(1, 8), Fraction(-5, 2), Fraction(0), Fraction(7)]
        w = to_array([encode_exact(Fraction(2), dt)] * 4, dt)
        b = to_array([encode_exact(v, dt) for v in bvals], dt)
        y, _, _, _ = impl_ln(to_array([c] * 4, dt).reshape(1, 4), w, b, None, 1e-5, dt)
        if [int(v) for v in bits_of(y, dt).reshape(-1)] != [encode_exact(v, dt) for v in bvals]:
            fails.append(f"ln constant row {dt}: y != b")
        a = Fraction(3, 2)
        x2 = to_array([encode_exact(a, dt), encode_exact(-a, dt)], dt).reshape(1, 2)
        y, _, _, _ = impl_ln(x2, None, None, None, 0.5, dt)
        q = a * a / (a * a + f32_exact(0.5))
        want = [exact.round_sqrt(1, q, dt), exact.round_sqrt(-1, q, dt)]
        if [int(v) for v in bits_of(y, dt).reshape(-1)] != want:
            fails.append(f"ln [a,-a] {dt}")
    return fails


def pin_ln_invariances(impl_ln):
    """With eps = 0: y(2^k x + c) == y(x) bit for bit for integer rows whose
    shifted and scaled values stay exact; and without affine, mean(n) = 0 and
    mean(n^2) = 1 in fp64."""
    fails = []
    rng = np.random.default_rng(55)
    for dt in ("bf16", "f32"):
        hidden = 64
        vals = rng.integers(-50, 51, size=(3, hidden)).astype(np.float64)
        vals[:, 0] = 60.0          # rows are never constant
        def enc(v):
            return to_array([encode_exact(Fraction(int(t)), dt) for t in v.reshape(-1)], dt).reshape(v.shape)
        base, _, n64, _ = impl_ln(enc(vals), None, None, None, 0.0, dt)
        for scale, shift in ((2, 0), (1, 64), (4, -32)):
            y2, _, _, _ = impl_ln(enc(vals * scale + shift), None, None, None, 0.0, dt)
            if not np.array_equal(bits_of(base, dt), bits_of(y2, dt)):
                fails.append(f"ln invariance {dt} scale={scale} shift={shift}")
        if n64 is None:
            fails.append("ln: no fp64 normalised values")
        else:
            if not (np.all(np.abs(n64.mean(axis=1)) < 1e-12) and np.all(np.abs((n64 ** 2).mean(axis=1) - 1) < 1e-12)):
                fails.append(f"ln moments {dt}")
    return fails


LN_PINS = [pin_ln_closed_forms, pin_ln_invariances, pin_ln_bruteforce]


# ----------------------------------------------------------------- MXFP8 pins
# impl_mx(x, w, residual, eps, dtype, weight_bias) -> (codes, scales, residual_out, v_exact)
# e4m3(v) -> codes ; e4m3_inv(codes) -> values.  Format: OCP FP8 E4M3 and MX v1.0.

def pin_e4m3_codec(e4m3, e4m3_inv):
    """Every code decodes to the value its bit fields define; every finite
    code encodes back to itself; the table's landmarks (448, 2^-6, 2^-9, 1, NaN)."""
    fails = []
    codes = np.arange(256, dtype=np.uint8)
    vals = e4m3_inv(codes)
    for c in range(256):
        want = exact.e4m3_decode(c)
        got = vals[c]
        if want is None:
            if not np.isnan(got):
                fails.append(f"e4m3 {c:#x} should be NaN")
        elif Fraction(float(got)) != want:
            fails.append(f"e4m3 {c:#x}: {got} != {float(want)}")
    finite = [c for c in range(256) if exact.e4m3_decode(c) is not None]
    back = e4m3(vals[finite])
    for c, b in zip(finite, back):
        if c != 0x80 and int(b) != c:
            fails.append(f"e4m3 round trip {c:#x} -> {int(b):#x}")
    for c, v in ((0x7E, 448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0x38, 1.0), (0x40, 2.0)):
        if vals[c] != v:
            fails.append(f"e4m3 landmark {c:#x}")
    return fails


def pin_e4m3_rounding(e4m3):
    """Midpoints between adjacent codes round to the even code; values just
    off a midpoint round to the nearer one; magnitudes above 448 saturate."""
    fails = []
    pts, want = [], []
    for c in range(0x00, 0x7E):
        a, b = exact.e4m3_decode(c), exact.e4m3_decode(c + 1)
        m = (a + b) / 2
        pts += [float(m), float(m) * (1 - 2 ** -40), float(m) * (1 + 2 ** -40)]
        want += [c if c % 2 == 0 else c + 1, c, c + 1]
    pts += [448.0, 463.9, 464.0, 500.0, 1e30, -1e30]
    want += [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    got = e4m3(np.array(pts, dtype=np.float64))
    for p, w_, g in zip(pts, want, got):
        if int(g) != w_:
            fails.append(f"e4m3({p!r}) = {int(g):#x}, want {w_:#x}")
    return fails


def pin_mx_bruteforce(impl_mx, n_cases=24, seed=909):
    """Random rows of 32 or 64 elements: codes and scales equal the exact
    rational answer (except values within 2^-44 of an E4M3 rounding midpoint)."""
    rng = np.random.default_rng(seed)
    fails = []
    for k in range(n_cases):
        dt = ("bf16", "f32")[k % 2]
        hidden = (32, 64)[(k // 2) % 2]
        has_w = bool((k // 4) % 2)
        has_res = bool((k // 8) % 2)
        b = (0.0, 1.0)[(k // 3) % 2] if has_w else 0.0
        eps = (0.0, 1e-6, 0.5)[k % 3]
        rows = 2
        lo_e, hi_e = ((-20, 20) if k % 5 == 0 else (-4, 4))     # some rows with a wide dynamic range
        xb = [random_bits(rng, dt, hidden, lo_e, hi_e) for _ in range(rows)]
        rb = [random_bits(rng, dt, hidden, -4, 4) for _ in range(rows)] if has_res else None
        wb = random_bits(rng, dt, hidden, -2, 2) if has_w else None
        x = to_array(sum(xb, []), dt).reshape(rows, hidden)
        res = to_array(sum(rb, []), dt).reshape(rows, hidden) if has_res else None
        w = to_array(wb, dt) if has_w else None
        codes, scales, _, _ = impl_mx(x, w, res, eps, dt, b)
        for r in range(rows):
            wc, ws, qs = exact.mxfp8_row_exact(xb[r], wb, rb[r] if has_res else None, f32_exact(eps), dt,
                                              Fraction(b))
            if [int(v) for v in scales[r]] != ws:
                fails.append(f"mx case {k} row {r}: scales {list(scales[r])} != {ws}")
                continue
            for i in range(hidden):
                if int(codes[r, i]) != wc[i]:
                    a, c2 = exact.e4m3_decode(int(codes[r, i]) & 0x7F), exact.e4m3_decode(wc[i] & 0x7F)
                    near = False
                    if a is not None and c2 is not None:
                        m2 = ((a + c2) / 2) ** 2
                        near = m2 > 0 and abs(qs[i] - m2) / m2 < Fraction(1, 2 ** 43)
                    if not near:
                        fails.append(f"mx case {k} ({dt}, H={hidden}) row {r} elem {i}: "
                                     f"{int(codes[r, i]):#x} != {wc[i]:#x}")
    return fails


def pin_mx_closed_forms(impl_mx):
    """A constant row with eps = 0 and no weight normalises to +-1 exactly:
    amax 1, scale 2^(0-8) (E8M0 code 119), every code E4M3(256) = 0x78 (sign
    kept).  Scaling a row by 2^k leaves codes and scales unchanged (eps = 0)."""
    fails = []
    for dt in ("bf16", "f32"):
        c = encode_exact(Fraction(-3, 2), dt)
        x = to_array([c] * 64, dt).reshape(1, 64)
        codes, scales, _, _ = impl_mx(x, None, None, 0.0, dt, 0.0)
        if [int(v) for v in scales[0]] != [119, 119] or any(int(v) != 0xF8 for v in codes[0]):
            fails.append(f"mx constant row {dt}: scales {list(scales[0])} codes {set(int(v) for v in codes[0])}")
        rng = np.random.default_rng(3)
        xb = random_bits(rng, dt, 64, -3, 3)
        x1 = to_array(xb, dt).reshape(1, 64)
        c1, s1, _, _ = impl_mx(x1, None, None, 0.0, dt, 0.0)
        xs = (x1.astype(np.float32) * np.float32(8.0)) if dt == "f32" else \
            ((((x1.astype(np.uint32) << 16).view(np.float32) * np.float32(8.0)).view(np.uint32)) >> 16).astype(np.uint16)
        c2, s2, _, _ = impl_mx(xs, None, None, 0.0, dt, 0.0)
        if not (np.array_equal(c1, c2) and np.array_equal(s1, s2)):
            fails.append(f"mx scale invariance {dt}")
    return fails


MX_PINS = [pin_mx_closed_forms, pin_mx_bruteforce]


# ----------------------------------------------------------------- NVFP4 pins
# impl_nv(x, w, residual, eps, dtype, weight_bias, tensor_scale) -> (codes packed, scales, residual_out, v_exact)

def unpack_nibbles(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def pin_e2m1_codec(e2m1, e2m1_inv):
    """The 16 codes decode to their definition's values; every midpoint rounds
    to the even code; magnitudes above 6 saturate."""
    fails = []
    vals = e2m1_inv(np.arange(16, dtype=np.uint8))
    for c in range(16):
        if Fraction(float(vals[c])) != exact.e2m1_decode(c):
            fails.append(f"e2m1 {c:#x}: {vals[c]}")
    pts, want = [], []
    for i in range(7):
        a, b = exact.E2M1_MAGS[i], exact.E2M1_MAGS[i + 1]
        m = float((a + b) / 2)
        pts += [m, m * (1 - 2 ** -40), m * (1 + 2 ** -40), -m]
        want += [i if i % 2 == 0 else i + 1, i, i + 1, 0x8 | (i if i % 2 == 0 else i + 1)]
    pts += [6.0, 6.9, 7.0, 1e9]
    want += [7, 7, 7, 7]
    got = e2m1(np.array(pts))
    for p, w_, g in zip(pts, want, got):
        if int(g) != w_:
            fails.append(f"e2m1({p}) = {int(g):#x}, want {w_:#x}")
    return fails


def pin_nv_bruteforce(impl_nv, n_cases=24, seed=707):
    """Random rows of 16 or 32 elements, several tensor scales: packed codes and
    scales equal the exact rational answer (except values within 2^-43 of a
    rounding midpoint)."""
    rng = np.random.default_rng(seed)
    fails = []
    for k in range(n_cases):
        dt = ("bf16", "f32")[k % 2]
        hidden = (16, 32)[(k // 2) % 2]
        has_w = bool((k // 4) % 2)
        has_res = bool((k // 8) % 2)
        S = (1.0, 0.125, 1.0 / 6.0, 3.0)[k % 4]
        b = 1.0 if (has_w and k % 3 == 0) else 0.0
        eps = (0.0, 1e-6, 0.5)[k % 3]
        rows = 2
        xb = [random_bits(rng, dt, hidden, -6, 6) for _ in range(rows)]
        rb = [random_bits(rng, dt, hidden, -4, 4) for _ in range(rows)] if has_res else None
        wb = random_bits(rng, dt, hidden, -2, 2) if has_w else None
        x = to_array(sum(xb, []), dt).reshape(rows, hidden)
        res = to_array(sum(rb, []), dt).reshape(rows, hidden) if has_res else None
        w = to_array(wb, dt) if has_w else None
        codes, scales, _, _ = impl_nv(x, w, res, eps, dt, b, S)
        codes = unpack_nibbles(codes)
        for r in range(rows):
            wc, ws, qs = exact.nvfp4_row_exact(xb[r], wb, rb[r] if has_res else None, f32_exact(eps), dt,
                                              Fraction(float(np.float32(S))), Fraction(b))
            if [int(v) for v in scales[r]] != ws:
                fails.append(f"nv case {k} row {r}: scales {list(scales[r])} != {ws}")
                continue
            for i in range(hidden):
                if int(codes[r, i]) != wc[i]:
                    lo, hi = sorted([int(codes[r, i]) & 7, wc[i] & 7])
                    near = False
                    if hi == lo + 1:
                        m2 = ((exact.E2M1_MAGS[lo] + exact.E2M1_MAGS[hi]) / 2) ** 2
                        near = abs(qs[i] - m2) / m2 < Fraction(1, 2 ** 43)
                    if not near:
                        fails.append(f"nv case {k} ({dt}, H={hidden}, S={S}) row {r} elem {i}: "
                                     f"{int(codes[r, i]):#x} != {wc[i]:#x}")
    return fails


def pin_nv_closed_forms(impl_nv):
    """A constant row with eps = 0 normalises to +-1; with tensor scale 1/6
    the block scale is E4M3(1) = 0x38 and every code is +-6 (0x7 / 0xF),
    packed low nibble first.  A zero row gives scale 0 and codes 0."""
    fails = []
    for dt in ("bf16", "f32"):
        S = float(np.float32(1.0 / 6.0))
        c = encode_exact(Fraction(-5, 4), dt)
        codes, scales, _, _ = impl_nv(to_array([c] * 32, dt).reshape(1, 32), None, None, 0.0, dt, 0.0, S)
        if [int(v) for v in scales[0]] != [0x38, 0x38] or any(int(v) != 0xFF for v in codes[0]):
            fails.append(f"nv constant row {dt}: {list(scales[0])} {list(codes[0])}")
        xs = to_array([encode_exact(Fraction(1), dt), encode_exact(Fraction(-1), dt)] * 8, dt)
        codes, scales, _, _ = impl_nv(xs.reshape(1, 16), None, None, 0.0, dt, 0.0, S)
        if [int(v) for v in codes[0]] != [0xF7] * 8:       # +6 (0x7) in the low nibble, -6 (0xF) high
            fails.append(f"nv nibble order {dt}: {list(codes[0])}")
        codes, scales, _, _ = impl_nv(to_array([0] * 16, dt).reshape(1, 16), None, None, 1e-5, dt, 0.0, 1.0)
        if int(scales[0, 0]) != 0 or any(int(v) != 0 for v in codes[0]):
            fails.append(f"nv zero row {dt}")
    return fails


NV_PINS = [pin_nv_closed_forms, pin_nv_bruteforce]


# ---------------------------------------------------------------- cast order

CAST_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "cast_order.txt")


def parse_cast_golden(path=CAST_GOLDEN):
    cases, cur = [], None
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "case":
            cur = {"name": rest[0]}
            cases.append(cur)
        elif key == "dtype":
            cur["dtype"] = rest[0]
        elif key == "eps":
            cur["eps"] = Fraction(rest[0])
        elif key in ("x", "w", "residual", "y", "plain", "resout"):
            cur[key] = None if rest == ["-"] else [Fraction(t) for t in _expand(rest)]
        else:
            raise ValueError(f"unknown key {key!r} in {path}")
    return cases


def pin_cast_golden(impl_cast):
    """Hand-derived cases in tests/golden/cast_order.txt, chosen so that the
    two-rounding order and the single rounding differ."""
    fails = []
    for c in parse_cast_golden():
        dt = c["dtype"]
        n = len(c["x"])
        enc = lambda vals: to_array([encode_exact(v, dt) for v in vals], dt)
        x = enc(c["x"]).reshape(1, n)
        w = None if c["w"] is None else enc(c["w"])
        res = None if c["residual"] is None else enc(c["residual"]).reshape(1, n)
        y, rout, _ = impl_cast(x, w, res, float(c["eps"]), dt)
        want = [encode_exact(v, dt) for v in c["y"]]
        got = [int(b) for b in bits_of(y, dt).reshape(-1)]
        if got != want:
            fails.append(f"cast golden {c['name']}: y bits {got} != {want}")
        if c.get("resout") is not None:
            got_r = [int(b) for b in bits_of(rout, dt).reshape(-1)]
            if got_r != [encode_exact(v, dt) for v in c["resout"]]:
                fails.append(f"cast golden {c['name']}: residual_out {got_r}")
    return fails


def pin_cast_bruteforce(impl_cast, n_cases=60, seed=2468):
    """Random tiny rows against the exact two-rounding answer.  The first
    rounding may go to the other neighbour only where the exact normalised
    value lies within 2^-44 (relative) of a rounding midpoint."""
    rng = np.random.default_rng(seed)
    fails = []
    eps_choices = [0.0, 1e-6, 1e-5, 0.25, 3.0]
    for k in range(n_cases):
        dt = ("bf16", "f32")[k % 2]
        has_w = (k // 2) % 4 != 0          # most cases with a weight: that is where the orders differ
        has_res = bool((k // 8) % 2)
        hidden = int(rng.integers(1, 9))
        rows = 3
        eps = eps_choices[k % len(eps_choices)]
        xb = [random_bits(rng, dt, hidden) for _ in range(rows)]
        rb = [random_bits(rng, dt, hidden) for _ in range(rows)] if has_res else None
        wb = random_bits(rng, dt, hidden, -2, 2) if has_w else None
        x = to_array(sum(xb, []), dt).reshape(rows, hidden)
        res = to_array(sum(rb, []), dt).reshape(rows, hidden) if has_res else None
        w = to_array(wb, dt) if has_w else None
        y, rout, _ = impl_cast(x, w, res, eps, dt)
        yb = bits_of(y, dt).reshape(rows, hidden)
        for r in range(rows):
            want, want_h, n_bits, qs, _ = exact.rmsnorm_cast_row_exact(
                xb[r], wb, rb[r] if has_res else None, f32_exact(eps), dt)
            for i in range(hidden):
                if int(yb[r, i]) == want[i]:
                    continue
                d = exact.midpoint_distance(qs[i], dt)
                alt = [exact.cast_times_weight(nb, wb[i], dt) if has_w else nb
                       for nb in exact.neighbours(n_bits[i], dt)]
                if d is None or d > Fraction(1, 2 ** 44) or int(yb[r, i]) not in alt:
                    fails.append(f"cast bruteforce case {k} ({dt}, w={has_w}, res={has_res}, H={hidden}, "
                                 f"eps={eps}) row {r} elem {i}: {int(yb[r, i]):#x} != {want[i]:#x}")
            if has_res:
                got_h = [int(b) for b in bits_of(rout, dt).reshape(rows, hidden)[r]]
                if got_h != want_h:
                    fails.append(f"cast bruteforce case {k}: residual_out row {r} {got_h} != {want_h}")
    return fails


def pin_cast_power_of_two_weight(impl_cast, seed=1357):
    """With weights +-2^k the weight multiply is exact, so the output is the
    unweighted output times the weight (both dtypes, rows of 300)."""
    rng = np.random.default_rng(seed)
    fails = []
    for dt in ("bf16", "f32"):
        rows, hidden = 4, 300
        x = to_array(random_bits(rng, dt, rows * hidden), dt).reshape(rows, hidden)
        wv = rng.choice([-4.0, -1.0, -0.5, 0.25, 1.0, 2.0, 8.0], hidden)
        w = to_array([encode_exact(Fraction(v), dt) for v in wv], dt)
        y0, _, _ = impl_cast(x, None, None, 1e-6, dt)
        y1, _, _ = impl_cast(x, w, None, 1e-6, dt)
        d0 = exact_values(y0, dt)
        d1 = exact_values(y1, dt)
        if not np.array_equal(d0 * wv[None, :], d1):
            fails.append(f"cast power-of-two weight ({dt}): y(w) != y(no w) * w")
    return fails


def exact_values(a, dt):
    """fp64 values of an I/O-type array (exact)."""
    if dt == "bf16":
        return (np.asarray(a, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


CAST_PINS = [pin_cast_golden, pin_cast_power_of_two_weight, pin_cast_bruteforce]


ALL_PINS = [pin_golden, pin_bruteforce, pin_constant_row, pin_scale_invariance,
            pin_unit_rms, pin_special_values, pin_single_element, pin_row_independence,
            pin_eps_dominated, pin_near_ties]
