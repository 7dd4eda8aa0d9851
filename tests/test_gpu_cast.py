"""RMSNorm in the op-by-op cast order (``rmsnorm_fwd_cast``) against the oracle.

The normalised value is rounded to the I/O type before the weight multiply
("model-as-a-kernel", sections "Method" and "Correctness"; the order itself is
the reading stated in the oracle).  bf16 outputs are bit-exact except where
the normalised value lies within the fp32 error bound of a bf16 rounding
midpoint (``parity.compare_cast_bf16``); fp32 outputs use the fp32 tolerance
and are the same bits as ``rmsnorm_fwd``, which runs the same arithmetic.
Every kernel family is forced through its plans: register (all threads x
chunks), bulk-copy (each piece size) and two-pass.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import parity
from row_reduction_norm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import row_reduction_norm_gb300 as R
    from test_gpu_parity import all_plans

THREADS = os.cpu_count() or 1
DEV = "cuda"


def cast_ref(x, r, w, eps, dtype, rows=None):
    xn, rn, wn = W.to_numpy_bits(x), W.to_numpy_bits(r), W.to_numpy_bits(w)
    if rows is not None:
        xn = xn[rows]
        rn = None if rn is None else rn[rows]
    return oracle.rmsnorm_cast(xn, w=wn, residual=rn, eps=eps, dtype=dtype, threads=THREADS), wn


def check_cast(y, h, x, r, w, eps, dtype, rows=None, what=""):
    (yr, hr, n64), wn = cast_ref(x, r, w, eps, dtype, rows)
    yg = W.to_numpy_bits(y)
    hg = W.to_numpy_bits(h)
    if rows is not None:
        yg = yg[rows]
        hg = None if hg is None else hg[rows]
    if dtype == "bf16":
        ok, rep = parity.compare_cast_bf16(yg, n64, wn, oracle.bf16_from_double)
    else:
        ok, rep = parity.compare_y(yg, yr, dtype)
    assert ok, f"{what}: y differs from the cast-order oracle: {rep}"
    if r is not None:
        assert parity.bits_equal(hg, hr), f"{what}: residual_out is not bit-exact"
    return rep


SWEEP = [(131, 576), (37, 128), (9, 4096), (3, 2048), (2, 16384), (19, 8), (2, 32768), (2, 40960)]


@pytest.mark.parametrize("rows,hidden", SWEEP)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_every_plan_matches_cast_oracle(rows, hidden, dtype):
    wl = W.Workload("cast", dtype, rows, hidden, 1e-5, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=hidden * 3 + rows, device=DEV)
    plans = all_plans(rows, hidden, R.dtype_code(x.dtype), True, odd_ch=True, tma=True)
    assert plans
    for p in plans:
        y, h = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=p, cast_before_weight=True)
        y1 = R.rms_norm(x, w=w, eps=wl.eps, plan=p, cast_before_weight=True)
        torch.cuda.synchronize()
        check_cast(y, h, x, r, w, wl.eps, dtype, what=f"plan {p.as_dict()}")
        check_cast(y1, None, x, None, w, wl.eps, dtype, what=f"plan {p.as_dict()} (no residual)")
        if dtype == "f32":
            yp = R.rms_norm(x, w=w, eps=wl.eps, plan=p)
            torch.cuda.synchronize()
            assert torch.equal(yp, y1), f"plan {p.as_dict()}: fp32 cast order is not the plain op's bits"


@pytest.mark.parametrize("hidden", [8, 576, 2048, 12288, 40960, 65536])
def test_without_weight_is_the_plain_op(hidden):
    wl = W.Workload("cast_nw", "bf16", 5, hidden, 1e-6, 1.0, 1.0, None)
    x, r, _ = W.make_inputs(wl, seed=hidden, device=DEV)
    y, h = R.rms_norm(x, residual=r, eps=wl.eps, cast_before_weight=True)
    yp, hp = R.rms_norm(x, residual=r, eps=wl.eps)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), yp.view(torch.int16))
    assert torch.equal(h.view(torch.int16), hp.view(torch.int16))


FULL = ["bf16_4096x576", "bf16_res_16384x2048", "bf16_res_4096x40960_w"]


@pytest.mark.parametrize("name", FULL)
def test_workload_library_plan(name):
    wl = W.WORKLOADS[name]
    rows = wl.rows if wl.rows * wl.hidden <= (1 << 25) else 64
    x, r, w = W.make_inputs(wl, seed=1, device=DEV, rows=rows)
    w = w if w is not None else torch.ones(wl.hidden, dtype=x.dtype, device=DEV)
    out = R.rms_norm(x, w=w, residual=r, eps=wl.eps, cast_before_weight=True)
    y, h = out if r is not None else (out, None)
    torch.cuda.synchronize()
    rep = check_cast(y, h, x, r, w, wl.eps, wl.dtype, what=name)
    assert rep["n_boundary"] < rep["n"] // 50


@pytest.mark.parametrize("name", ["bf16_2048x65536_w", "bf16_res_2048x65536_w"])
def test_long_rows_full_size_sampled(name):
    # the bulk-copy kernel (no residual) and the two-pass kernel (residual) at full size
    wl = W.WORKLOADS[name]
    x, r, w = W.make_inputs(wl, seed=2, device=DEV)
    out = R.rms_norm(x, w=w, residual=r, eps=wl.eps, cast_before_weight=True)
    y, h = out if r is not None else (out, None)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 777, wl.rows // 2, wl.rows - 2, wl.rows - 1])
    check_cast(y, h, x, r, w, wl.eps, wl.dtype, rows=rows, what=name)
    del x, r, w, y, h, out
    torch.cuda.empty_cache()


def test_orders_differ_and_batch_invariant():
    # the two orders give different bf16 bits on ordinary data, and a row's
    # cast-order result does not depend on the rows launched with it
    wl = W.WORKLOADS["bf16_res_16384x2048"]
    x, r, w = W.make_inputs(wl, seed=4, device=DEV, rows=4096)
    y, _ = R.rms_norm(x, w=w, residual=r, eps=wl.eps, cast_before_weight=True)
    yp, _ = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    y7, _ = R.rms_norm(x[100:107].contiguous(), w=w, residual=r[100:107].contiguous(), eps=wl.eps,
                       cast_before_weight=True)
    torch.cuda.synchronize()
    differ = int((y.view(torch.int16) != yp.view(torch.int16)).sum())
    assert differ > 0
    assert torch.equal(y7.view(torch.int16), y[100:107].view(torch.int16))


def test_argument_checks():
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.ones(64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        R.rms_norm(x, w=w, cast_before_weight=True, weight_bias=1.0)
    from row_reduction_norm_gb300 import _native as N
    y = torch.empty_like(x)
    assert N.rmsnorm_fwd_cast_status(x.data_ptr(), None, w.data_ptr(), y.data_ptr(), None, 4, 64, -1.0,
                                     N.RMSNORM_BF16) == N.RMSNORM_EINVAL
    assert N.rmsnorm_fwd_cast_status(x.data_ptr(), None, w.data_ptr(), y.data_ptr(), None, 0, 64, 1e-6,
                                     N.RMSNORM_BF16) == N.RMSNORM_OK


@pytest.mark.parametrize("hidden", [576, 4096, 40960])
def test_misaligned_and_in_place(hidden):
    # pointers one element off 16 bytes take the scalar two-pass kernel; y may be x
    wl = W.Workload("cast_odd", "bf16", 7, hidden, 1e-6, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=hidden + 1, device=DEV)

    def shifted(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
        v = buf[1:].view(t.shape)
        v.copy_(t)
        return v

    xs, rs, ws = shifted(x), shifted(r), shifted(w)
    y, h = R.rms_norm(xs, w=ws, residual=rs, eps=wl.eps, cast_before_weight=True)
    torch.cuda.synchronize()
    check_cast(y, h, x, r, w, wl.eps, "bf16", what=f"misaligned H={hidden}")
    xi = x.clone()
    R.rms_norm(xi, w=w, eps=wl.eps, out=xi, cast_before_weight=True)
    torch.cuda.synchronize()
    check_cast(xi, None, x, None, w, wl.eps, "bf16", what=f"in place H={hidden}")


def test_golden_cases_through_the_kernel():
    # the hand-derived cases of tests/golden/cast_order.txt, through the C ABI;
    # bf16 bit-exact (no case lies near a first-rounding midpoint), fp32 within
    # the fp32 tolerance
    import pins
    for c in pins.parse_cast_golden():
        dt = c["dtype"]
        n = len(c["x"])
        enc = lambda vals: pins.to_array([pins.encode_exact(v, dt) for v in vals], dt)
        tdt = W.TORCH_DTYPE[dt]

        def dev(a, shape):
            t = torch.from_numpy(a.astype(a.dtype).reshape(shape).copy())
            return (t.view(torch.bfloat16) if dt == "bf16" else t).to(DEV)

        x = dev(enc(c["x"]), (1, n))
        w = dev(enc(c["w"]), (n,))
        r = None if c["residual"] is None else dev(enc(c["residual"]), (1, n))
        out = R.rms_norm(x, w=w, residual=r, eps=float(c["eps"]), cast_before_weight=True)
        y, h = out if r is not None else (out, None)
        torch.cuda.synchronize()
        assert y.dtype == tdt
        want = enc(c["y"]).reshape(1, n)
        got = W.to_numpy_bits(y)
        if dt == "bf16":
            assert np.array_equal(got, want), f"{c['name']}: {got} != {want}"
        else:
            ok, rep = parity.compare_y(got, want, dt)
            assert ok, f"{c['name']}: {rep}"
        if c.get("resout") is not None:
            assert np.array_equal(W.to_numpy_bits(h), enc(c["resout"]).reshape(1, n)), c["name"]
