"""GPU parity of the fused LayerNorm against the oracle, through the C ABI
(GB300 only).  Tolerance: ``parity.compare_ln`` (a bound on the terms of
w * n + b, derived in parity.py); residual_out bit-exact."""
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
    from row_reduction_norm_gb300 import _native as N
    from test_gpu_parity import all_plans

THREADS = os.cpu_count() or 1
DEV = "cuda"


def ln_check(y, h, x, r, w, b, eps, dtype, what):
    xn, rn = W.to_numpy_bits(x), W.to_numpy_bits(r)
    wn, bn = W.to_numpy_bits(w), W.to_numpy_bits(b)
    yr, hr, n64, y64 = oracle.layernorm(xn, w=wn, b=bn, residual=rn, eps=eps, dtype=dtype, want_exact=True,
                                        threads=THREADS)
    src = hr if rn is not None else xn
    hv = parity.decode(src, dtype)
    mean_abs = np.abs(hv).mean(axis=1)
    var = ((hv - hv.mean(axis=1, keepdims=True)) ** 2).mean(axis=1)
    sigma = np.sqrt(var + float(np.float32(eps)))
    ok, rep = parity.compare_ln(W.to_numpy_bits(y), y64, n64, wn, bn, mean_abs, sigma, dtype)
    assert ok, f"{what}: {rep}"
    if r is not None:
        assert parity.bits_equal(W.to_numpy_bits(h), hr), f"{what}: residual_out not bit-exact"
    return rep


@pytest.mark.parametrize("name", list(W.LN_WORKLOADS))
def test_ln_workload_full_size(name):
    wl = W.LN_WORKLOADS[name]
    x, r, w, b = W.make_ln_inputs(wl, device=DEV)
    out = R.layer_norm(x, w=w, b=b, residual=r, eps=wl.eps)
    y, h = out if r is not None else (out, None)
    torch.cuda.synchronize()
    ln_check(y, h, x, r, w, b, wl.eps, wl.dtype, name)


LN_SWEEP = [(131, 768), (9, 4096), (37, 128), (5, 8192), (3, 2048), (2, 16384), (19, 64)]


@pytest.mark.parametrize("rows,hidden", LN_SWEEP)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ln_every_plan(rows, hidden, dtype):
    wl = W.Workload("ln-sweep", dtype, rows, hidden, 1e-5, 1.0, 1.0, 0.1, b_std=0.1, x_mean=0.25)
    x, r, w, b = W.make_ln_inputs(wl, seed=rows + hidden, device=DEV)
    code = R.dtype_code(x.dtype)
    plans = [p for p in all_plans(rows, hidden, code, True, odd_ch=True, min_block=128)
             if p.kernel == N.RMSNORM_KERNEL_LOOP or p.threads_per_row <= 256]
    for p in plans:
        for ww, bb, rr in ((w, b, r), (w, None, None), (None, None, r)):
            out = R.layer_norm(x, w=ww, b=bb, residual=rr, eps=wl.eps, plan=p)
            y, h = out if rr is not None else (out, None)
            torch.cuda.synchronize()
            ln_check(y, h, x, rr, ww, bb, wl.eps, dtype, f"plan {p.as_dict()} w={ww is not None} "
                                                           f"b={bb is not None} res={rr is not None}")


@pytest.mark.parametrize("hidden", [1, 2, 7, 33, 768, 1000, 1025, 4096, 12288, 32768, 65536])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ln_tail_sweep(hidden, dtype):
    for rows in (1, 3, 67):
        wl = W.Workload("ln-tail", dtype, rows, hidden, 1e-5, 1.0, 1.0, 0.1, b_std=0.1)
        x, r, w, b = W.make_ln_inputs(wl, seed=rows * 3 + hidden, device=DEV)
        y, h = R.layer_norm(x, w=w, b=b, residual=r, eps=wl.eps)
        torch.cuda.synchronize()
        ln_check(y, h, x, r, w, b, wl.eps, dtype, f"H={hidden} rows={rows}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ln_constant_rows_give_bias(dtype):
    tdt = W.TORCH_DTYPE[dtype]
    x = torch.full((8, 768), 0.75, device=DEV, dtype=tdt)
    w = torch.full((768,), 2.0, device=DEV, dtype=tdt)
    b = W.random_rows(dtype, 1, 768, seed=3, device=DEV).reshape(-1)
    y = R.layer_norm(x, w=w, b=b, eps=1e-5)
    torch.cuda.synchronize()
    assert torch.equal(y, b.expand_as(y))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ln_large_mean_offset(dtype):
    """Rows whose mean is 100x their spread: the term bound covers the mean's rounding."""
    wl = W.Workload("ln-offset", dtype, 64, 2048, 1e-5, 1.0, None, 0.1, b_std=0.1, x_mean=100.0)
    x, _, w, b = W.make_ln_inputs(wl, seed=11, device=DEV)
    y = R.layer_norm(x, w=w, b=b, eps=wl.eps)
    torch.cuda.synchronize()
    ln_check(y, None, x, None, w, b, wl.eps, dtype, "offset")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ln_misaligned_in_place_deterministic(dtype):
    tdt = W.TORCH_DTYPE[dtype]
    rows, hidden = 21, 1536
    buf = W.random_rows(dtype, 1, rows * hidden + 1, seed=6, device=DEV).reshape(-1)
    x = buf[1:].view(rows, hidden)
    w = (1 + 0.1 * W.random_rows(dtype, 1, hidden, seed=7, device=DEV)).to(tdt).reshape(-1)
    p = R.layer_norm_plan_for(x, w=w)
    assert p.vec_elems == 1 and p.kernel == N.RMSNORM_KERNEL_LOOP
    ref = x.clone()
    y1 = R.layer_norm(x, w=w, eps=1e-5)
    y2 = R.layer_norm(x, w=w, eps=1e-5)
    R.layer_norm(x, w=w, eps=1e-5, out=x)   # in place
    torch.cuda.synchronize()
    assert parity.bits_equal(W.to_numpy_bits(y1), W.to_numpy_bits(y2))
    assert parity.bits_equal(W.to_numpy_bits(x), W.to_numpy_bits(y1))
    ln_check(y1, None, ref, None, w, None, 1e-5, dtype, "misaligned")


def test_ln_status_codes():
    x = torch.zeros((4, 64), device=DEV, dtype=torch.bfloat16)
    y = torch.empty_like(x)
    b = torch.zeros(64, device=DEV, dtype=torch.bfloat16)
    assert N.layernorm_fwd_status(x.data_ptr(), None, None, b.data_ptr(), y.data_ptr(), None, 4, 64, 1e-5, 1) \
        == N.RMSNORM_EINVAL      # bias without weight
    assert N.layernorm_fwd_status(x.data_ptr(), None, None, None, y.data_ptr(), None, 4, 64, -1.0, 1) \
        == N.RMSNORM_EINVAL
    assert N.layernorm_fwd_status(x.data_ptr(), None, None, None, y.data_ptr(), None, 4, 64, 1e-5, 1) \
        == N.RMSNORM_OK
    torch.cuda.synchronize()
