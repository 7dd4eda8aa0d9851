"""The oracle pinned to facts other than itself (CPU only).

Every pin in ``pins.py`` must hold for the oracle; every planted mistake in
``mutants.py`` must be caught by at least one pin; and an independent numpy
restatement of the definition must agree with the oracle bit for bit on
seeded inputs shaped like the workloads.
"""
import numpy as np
import pytest

import mutants
import oracle
import pins
from row_reduction_norm_gb300 import workloads as W


def oracle_impl(x, w, residual, eps, dtype):
    return oracle.rmsnorm(x, w=w, residual=residual, eps=eps, dtype=dtype, want_exact=True)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    assert pin(oracle_impl) == []


def test_oracle_bruteforce_many():
    assert pins.pin_bruteforce(oracle_impl, n_cases=600, seed=99) == []


def test_numpy_restatement_passes_pins():
    impl = lambda x, w, r, e, d: mutants.reference(x, w, r, e, d)
    for pin in pins.ALL_PINS:
        assert pin(impl) == [], pin.__name__


@pytest.mark.parametrize("mistake", mutants.MISTAKES)
def test_pins_catch_planted_mistake(mistake):
    impl = lambda x, w, r, e, d: mutants.reference(x, w, r, e, d, mistake=mistake)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            fails = pin(impl)
        except Exception as ex:  # a crash also counts as caught
            fails = [repr(ex)]
        if fails:
            caught.append(pin.__name__)
            break   # one catching pin is enough; the pins are ordered cheapest first
    assert caught, f"no pin catches the planted mistake {mistake!r}"


@pytest.mark.parametrize("name", ["f32_64x256", "bf16_4096x576", "bf16_res_16384x2048",
                                  "bf16_res_65536x8192_nw"])
def test_oracle_matches_numpy_restatement(name):
    wl = W.WORKLOADS[name]
    rows = min(wl.rows, 256)
    x, r, w = W.make_inputs(wl, seed=3, rows=rows)
    xn, rn, wn = W.to_numpy_bits(x), W.to_numpy_bits(r), W.to_numpy_bits(w)
    y, h, _ = oracle.rmsnorm(xn, w=wn, residual=rn, eps=wl.eps, dtype=wl.dtype)
    y2, h2, _ = mutants.reference(xn, wn, rn, wl.eps, wl.dtype)
    assert np.array_equal(pins.bits_of(y, wl.dtype), pins.bits_of(y2, wl.dtype))
    if rn is not None:
        assert np.array_equal(pins.bits_of(h, wl.dtype), pins.bits_of(h2, wl.dtype))


def test_oracle_threads_match_single_thread():
    wl = W.WORKLOADS["bf16_res_16384x2048"]
    x, r, w = W.make_inputs(wl, seed=5, rows=300)
    xn, rn, wn = W.to_numpy_bits(x), W.to_numpy_bits(r), W.to_numpy_bits(w)
    a = oracle.rmsnorm(xn, w=wn, residual=rn, eps=wl.eps, dtype="bf16", threads=1)
    b = oracle.rmsnorm(xn, w=wn, residual=rn, eps=wl.eps, dtype="bf16", threads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bf16_conversion_definition():
    # every bf16 encoding decodes to the value of its fp32 extension and rounds back to itself
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.double_from_bf16(bits)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    same = (vals == ref) | (np.isnan(vals) & np.isnan(ref))
    assert same.all()
    finite = ~np.isnan(vals)
    back = oracle.bf16_from_double(vals[finite])
    assert np.array_equal(back, bits[finite])


def oracle_impl_b(x, w, residual, eps, dtype, weight_bias):
    if weight_bias is None:
        return oracle.rmsnorm(x, w=w, residual=residual, eps=eps, dtype=dtype, want_exact=True)
    return oracle.rmsnorm(x, w=w, residual=residual, eps=eps, dtype=dtype, want_exact=True,
                          weight_bias=weight_bias)


def oracle_impl_qk(x, qh, kh, hd, q_w, k_w, eps, dtype, weight_bias):
    return oracle.rmsnorm_qk(x, qh, kh, hd, q_w=q_w, k_w=k_w, eps=eps, dtype=dtype, weight_bias=weight_bias)


def test_oracle_weight_bias_pin():
    assert pins.pin_weight_bias(oracle_impl_b) == []


def test_oracle_qk_pin():
    assert pins.pin_qk_heads(oracle_impl_qk) == []


def test_restatement_passes_bias_and_qk_pins():
    assert pins.pin_weight_bias(lambda x, w, r, e, d, b: mutants.reference(x, w, r, e, d, weight_bias=b)) == []
    assert pins.pin_qk_heads(lambda x, qh, kh, hd, qw, kw, e, d, b:
                             mutants.reference_qk(x, qh, kh, hd, qw, kw, e, d, weight_bias=b)) == []


@pytest.mark.parametrize("mistake", mutants.BIAS_MISTAKES)
def test_weight_bias_pin_catches(mistake):
    impl = lambda x, w, r, e, d, b: mutants.reference(x, w, r, e, d, mistake=mistake, weight_bias=b)
    assert pins.pin_weight_bias(impl) != []


@pytest.mark.parametrize("mistake", mutants.QK_MISTAKES)
def test_qk_pin_catches(mistake):
    impl = lambda x, qh, kh, hd, qw, kw, e, d, b: mutants.reference_qk(x, qh, kh, hd, qw, kw, e, d,
                                                                       weight_bias=b, mistake=mistake)
    assert pins.pin_qk_heads(impl) != []



def oracle_impl_ln(x, w, b, residual, eps, dtype):
    return oracle.layernorm(x, w=w, b=b, residual=residual, eps=eps, dtype=dtype, want_exact=True)


@pytest.mark.parametrize("pin", pins.LN_PINS, ids=lambda p: p.__name__)
def test_oracle_ln_pin(pin):
    assert pin(oracle_impl_ln) == []


def test_ln_restatement_passes_pins():
    impl = lambda x, w, b, r, e, d: mutants.reference_ln(x, w, b, r, e, d)
    for pin in pins.LN_PINS:
        assert pin(impl) == [], pin.__name__


@pytest.mark.parametrize("mistake", mutants.LN_MISTAKES)
def test_ln_pins_catch_planted_mistake(mistake):
    impl = lambda x, w, b, r, e, d: mutants.reference_ln(x, w, b, r, e, d, mistake=mistake)
    caught = [p.__name__ for p in pins.LN_PINS if p(impl)]
    assert caught, mistake


def test_ln_oracle_matches_restatement_on_workload_shapes():
    from row_reduction_norm_gb300 import workloads as W
    for dt, h in (("bf16", 768), ("f32", 1024), ("bf16", 4096)):
        x = W.to_numpy_bits(W.random_rows(dt, 64, h, seed=h, std=3.0))
        wv = W.to_numpy_bits(W.random_rows(dt, 1, h, seed=h + 1).reshape(-1))
        bv = W.to_numpy_bits(W.random_rows(dt, 1, h, seed=h + 2).reshape(-1))
        y1 = oracle.layernorm(x, w=wv, b=bv, eps=1e-5, dtype=dt)[0]
        y2 = mutants.reference_ln(x, wv, bv, None, 1e-5, dt)[0]
        assert np.array_equal(pins.bits_of(y1, dt), pins.bits_of(y2, dt))



def oracle_impl_mx(x, w, residual, eps, dtype, weight_bias):
    return oracle.rmsnorm_mxfp8(x, w=w, residual=residual, eps=eps, dtype=dtype, weight_bias=weight_bias)


def test_oracle_e4m3_codec_and_rounding():
    assert pins.pin_e4m3_codec(oracle.e4m3_from_double, oracle.double_from_e4m3) == []
    assert pins.pin_e4m3_rounding(oracle.e4m3_from_double) == []


@pytest.mark.parametrize("pin", pins.MX_PINS, ids=lambda p: p.__name__)
def test_oracle_mx_pin(pin):
    assert pin(oracle_impl_mx) == []


def test_mx_restatement_passes_pins_and_matches_oracle():
    impl = lambda x, w, r, e, d, b: mutants.reference_mx(x, w, r, e, d, weight_bias=b)
    for pin in pins.MX_PINS:
        assert pin(impl) == [], pin.__name__
    assert pins.pin_e4m3_rounding(lambda v: mutants._e4m3(v)) == []
    from row_reduction_norm_gb300 import workloads as W
    x = W.to_numpy_bits(W.random_rows("bf16", 64, 2048, seed=5))
    a = oracle.rmsnorm_mxfp8(x, eps=1e-6, dtype="bf16")
    b = mutants.reference_mx(x, None, None, 1e-6, "bf16")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("mistake", mutants.MX_MISTAKES)
def test_mx_pins_catch_planted_mistake(mistake):
    impl = lambda x, w, r, e, d, b: mutants.reference_mx(x, w, r, e, d, weight_bias=b, mistake=mistake)
    caught = [p.__name__ for p in pins.MX_PINS if p(impl)]
    if not caught and mistake in ("truncate_codes", "ties_away_codes", "no_saturation"):
        # rounding-rule mistakes also show on the bare encoder's midpoints
        enc = lambda v: mutants._e4m3(v, mode={"truncate_codes": "trunc", "ties_away_codes": "away"}.get(
            mistake, "rne"), saturate=mistake != "no_saturation")
        caught = ["pin_e4m3_rounding"] if pins.pin_e4m3_rounding(enc) else []
    assert caught, mistake


def test_compare_helpers_flag_planted_differences():
    """The GPU-side comparison helpers accept the oracle against itself and
    reject a flipped code, a shifted scale and a 2-ulp bf16 difference."""
    import parity
    from row_reduction_norm_gb300 import workloads as W
    x = W.to_numpy_bits(W.random_rows("bf16", 16, 576, seed=1))
    co, so, _, v = oracle.rmsnorm_mxfp8(x, eps=1e-5, dtype="bf16")
    assert parity.compare_mx(co, so, co, so, v, oracle.e4m3_from_double)[0]
    c2 = co.copy()
    c2[3, 7] ^= 1
    assert not parity.compare_mx(c2, so, co, so, v, oracle.e4m3_from_double)[0]
    s2 = so.copy()
    s2[2, 1] += 1
    assert not parity.compare_mx(co, s2, co, so, v, oracle.e4m3_from_double)[0]
    y, _, _ = oracle.rmsnorm(x, eps=1e-5, dtype="bf16")
    assert parity.compare_y(y, y, "bf16")[0]
    y2 = y.copy()
    y2[0, 0] += 2
    assert not parity.compare_y(y2, y, "bf16")[0]



def oracle_impl_nv(x, w, residual, eps, dtype, weight_bias, tensor_scale):
    return oracle.rmsnorm_nvfp4(x, w=w, residual=residual, eps=eps, dtype=dtype, weight_bias=weight_bias,
                                tensor_scale=tensor_scale)


def test_oracle_e2m1_codec():
    assert pins.pin_e2m1_codec(oracle.e2m1_from_double, oracle.double_from_e2m1) == []


@pytest.mark.parametrize("pin", pins.NV_PINS, ids=lambda p: p.__name__)
def test_oracle_nv_pin(pin):
    assert pin(oracle_impl_nv) == []


def test_nv_restatement_passes_pins_and_matches_oracle():
    impl = lambda x, w, r, e, d, b, S: mutants.reference_nv(x, w, r, e, d, weight_bias=b, tensor_scale=S)
    for pin in pins.NV_PINS:
        assert pin(impl) == [], pin.__name__
    assert pins.pin_e2m1_codec(lambda v: mutants._e2m1(v), oracle.double_from_e2m1) == []
    from row_reduction_norm_gb300 import workloads as W
    x = W.to_numpy_bits(W.random_rows("bf16", 64, 2048, seed=6))
    a = oracle.rmsnorm_nvfp4(x, eps=1e-6, dtype="bf16", tensor_scale=0.25)
    b = mutants.reference_nv(x, None, None, 1e-6, "bf16", tensor_scale=0.25)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("mistake", mutants.NV_MISTAKES)
def test_nv_pins_catch_planted_mistake(mistake):
    impl = lambda x, w, r, e, d, b, S: mutants.reference_nv(x, w, r, e, d, weight_bias=b, tensor_scale=S,
                                                            mistake=mistake)
    caught = []
    for p in pins.NV_PINS:
        try:
            if p(impl):
                caught.append(p.__name__)
        except Exception as ex:   # a crash also counts as caught
            caught.append(f"{p.__name__}: {ex!r}")
    if not caught and mistake in ("nv_truncate", "nv_no_saturation"):
        enc = lambda v: mutants._e2m1(v, mode="trunc" if mistake == "nv_truncate" else "rne",
                                      saturate=mistake != "nv_no_saturation")
        caught = ["pin_e2m1_codec"] if pins.pin_e2m1_codec(enc, oracle.double_from_e2m1) else []
    assert caught, mistake



def test_compare_nv_flags_planted_differences():
    import parity
    from row_reduction_norm_gb300 import workloads as W
    x = W.to_numpy_bits(W.random_rows("bf16", 16, 512, seed=2))
    co, so, _, v = oracle.rmsnorm_nvfp4(x, eps=1e-5, dtype="bf16", tensor_scale=1 / 64)
    assert parity.compare_nv(co, so, co, so, v, 1 / 64, oracle.e2m1_from_double)[0]
    c2 = co.copy()
    c2[1, 3] ^= 0x02
    assert not parity.compare_nv(c2, so, co, so, v, 1 / 64, oracle.e2m1_from_double)[0]
    s2 = so.copy()
    s2[4, 2] += 1
    assert not parity.compare_nv(co, s2, co, so, v, 1 / 64, oracle.e2m1_from_double)[0]


# ---------------------------------------------------------------- cast order

def oracle_impl_cast(x, w, residual, eps, dtype):
    return oracle.rmsnorm_cast(x, w=w, residual=residual, eps=eps, dtype=dtype)


@pytest.mark.parametrize("pin", pins.CAST_PINS, ids=lambda p: p.__name__)
def test_oracle_cast_pin(pin):
    assert pin(oracle_impl_cast) == []


def test_cast_restatement_passes_pins():
    for pin in pins.CAST_PINS:
        assert pin(mutants.reference_cast) == [], pin.__name__


@pytest.mark.parametrize("mistake", mutants.CAST_MISTAKES)
def test_cast_pins_catch_planted_mistake(mistake):
    impl = lambda x, w, r, e, d: mutants.reference_cast(x, w, r, e, d, mistake=mistake)
    assert any(pin(impl) for pin in pins.CAST_PINS), f"no pin catches {mistake!r}"


def test_cast_golden_cases_discriminate():
    # the plain (single-rounding) oracle gives the "plain" column of every
    # cast-order golden case, so each case separates the two orders
    for c in pins.parse_cast_golden():
        if c.get("plain") is None:
            continue
        dt = c["dtype"]
        n = len(c["x"])
        enc = lambda vals: pins.to_array([pins.encode_exact(v, dt) for v in vals], dt)
        res = None if c["residual"] is None else enc(c["residual"]).reshape(1, n)
        y, _, _ = oracle.rmsnorm(enc(c["x"]).reshape(1, n), w=enc(c["w"]), residual=res,
                                 eps=float(c["eps"]), dtype=dt)
        assert [int(b) for b in pins.bits_of(y, dt).reshape(-1)] == [pins.encode_exact(v, dt) for v in c["plain"]]
        assert c["plain"] != c["y"]


@pytest.mark.parametrize("name", ["bf16_4096x576", "bf16_res_16384x2048", "f32_64x256"])
def test_cast_oracle_matches_restatement_and_plain_without_weight(name):
    wl = W.WORKLOADS[name]
    x, r, w = W.make_inputs(wl, seed=11, rows=min(wl.rows, 64))
    xn, rn, wn = W.to_numpy_bits(x), W.to_numpy_bits(r), W.to_numpy_bits(w)
    y, h, n64 = oracle.rmsnorm_cast(xn, w=wn, residual=rn, eps=wl.eps, dtype=wl.dtype, threads=3)
    y2, h2, v2 = mutants.reference_cast(xn, wn, rn, wl.eps, wl.dtype)
    assert np.array_equal(pins.bits_of(y, wl.dtype), pins.bits_of(y2, wl.dtype))
    if rn is not None:
        assert np.array_equal(pins.bits_of(h, wl.dtype), pins.bits_of(h2, wl.dtype))
    assert np.allclose(n64, v2, rtol=1e-13, atol=0)
    y0, _, _ = oracle.rmsnorm_cast(xn, residual=rn, eps=wl.eps, dtype=wl.dtype)
    yp, _, _ = oracle.rmsnorm(xn, residual=rn, eps=wl.eps, dtype=wl.dtype)
    assert np.array_equal(pins.bits_of(y0, wl.dtype), pins.bits_of(yp, wl.dtype))


def test_compare_cast_flags_planted_differences():
    import parity
    wl = W.WORKLOADS["bf16_res_16384x2048"]
    x, r, w = W.make_inputs(wl, seed=8, rows=64)
    xn, rn, wn = W.to_numpy_bits(x), W.to_numpy_bits(r), W.to_numpy_bits(w)
    y, _, n64 = oracle.rmsnorm_cast(xn, w=wn, residual=rn, eps=wl.eps, dtype="bf16")
    ok, rep = parity.compare_cast_bf16(y, n64, wn, oracle.bf16_from_double)
    assert ok and 0 < rep["n_boundary"] < rep["n"] // 100, rep
    yp, _, _ = oracle.rmsnorm(xn, w=wn, residual=rn, eps=wl.eps, dtype="bf16")
    ok, rep = parity.compare_cast_bf16(yp, n64, wn, oracle.bf16_from_double)
    assert not ok and rep["n_bad"] > 0           # the single rounding is a different result
    bad = y.copy()
    bad[3, 5] ^= 1
    assert not parity.compare_cast_bf16(bad, n64, wn, oracle.bf16_from_double)[0]


def test_cast_oracle_bruteforce_many():
    assert pins.pin_cast_bruteforce(oracle_impl_cast, n_cases=400, seed=4242) == []
