"""GPU parity of RMSNorm with NVFP4 output against the oracle, through the
C ABI (GB300 only).  Codes and scales must equal the oracle's except where
the exact value lies within the fp32 error of a decision boundary
(``parity.compare_nv``)."""
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


def nv_check(out, x, r, w, eps, S, what, weight_bias=0.0):
    codes, scales = out[0], out[1]
    co, so, ho, v64 = oracle.rmsnorm_nvfp4(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r),
                                           eps=eps, dtype="bf16", weight_bias=weight_bias, tensor_scale=S,
                                           threads=THREADS)
    ok, rep = parity.compare_nv(codes.cpu().numpy(), scales.cpu().numpy(), co, so, v64, S, oracle.e2m1_from_double)
    assert ok, f"{what}: {rep}"
    if r is not None:
        assert parity.bits_equal(W.to_numpy_bits(out[2]), ho), f"{what}: residual_out"
    return rep


@pytest.mark.parametrize("name", ["bf16_4096x576", "bf16_res_16384x2048", "bf16_qk_262144x128"])
@pytest.mark.parametrize("S", [1.0 / 64, 1.0, 0.3])
def test_nv_workloads(name, S):
    wl = W.WORKLOADS[name]
    x, r, w = W.make_inputs(wl, device=DEV)
    out = R.rms_norm_nvfp4(x, w=w, residual=r, eps=wl.eps, tensor_scale=S)
    torch.cuda.synchronize()
    rep = nv_check(out, x, r, w, wl.eps, S, name)
    assert rep["code_flips"] <= 1e-4 * x.numel()


@pytest.mark.parametrize("rows,hidden", [(37, 576), (9, 4096), (64, 128), (3, 16), (5, 2048), (2, 16384)])
def test_nv_every_plan(rows, hidden):
    wl = W.Workload("nv-sweep", "bf16", rows, hidden, 1e-5, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=rows + hidden, device=DEV)
    plans = [p for p in all_plans(rows, hidden, N.RMSNORM_BF16, True) if p.kernel == N.RMSNORM_KERNEL_REG]
    assert plans
    for p in plans:
        for ww, rr, b in ((w, r, 0.0), (None, None, 0.0), (w, None, 1.0)):
            out = R.rms_norm_nvfp4(x, w=ww, residual=rr, eps=wl.eps, weight_bias=b, tensor_scale=1.0 / 32, plan=p)
            torch.cuda.synchronize()
            nv_check(out, x, rr, ww, wl.eps, 1.0 / 32, f"plan {p.as_dict()} w={ww is not None} res={rr is not None}",
                     weight_bias=b)


def test_nv_special_blocks():
    x = W.random_rows("bf16", 5, 256, seed=9, device=DEV)
    x[0, 7] = float("nan")
    x[1, 100] = float("inf")
    x[2] = 0.0
    x[3, :16] = x[3, :16] * 1e-6
    out = R.rms_norm_nvfp4(x, eps=1e-5, tensor_scale=1.0 / 16)
    torch.cuda.synchronize()
    nv_check(out, x, None, None, 1e-5, 1.0 / 16, "special")
    codes, scales = out
    assert int(scales[0, 0]) == 0x7F and int(codes[0].max()) == 0
    assert int(scales[2].max()) == 0 and int(codes[2].max()) == 0


def test_nv_argument_checks():
    x = torch.zeros((4, 64), device=DEV, dtype=torch.bfloat16)
    c = torch.empty((4, 32), device=DEV, dtype=torch.uint8)
    s = torch.empty((4, 4), device=DEV, dtype=torch.uint8)
    st = N.rmsnorm_fwd_nvfp4_status
    assert st(x.data_ptr(), None, None, c.data_ptr(), s.data_ptr(), None, 4, 64, 1e-6, 0.0, 1.0, 1) == N.RMSNORM_OK
    assert st(x.data_ptr(), None, None, c.data_ptr(), s.data_ptr(), None, 4, 40, 1e-6, 0.0, 1.0, 1) \
        == N.RMSNORM_EINVAL                                           # hidden not a multiple of 16
    assert st(x.data_ptr(), None, None, c.data_ptr(), s.data_ptr(), None, 4, 64, 1e-6, 0.0, 0.0, 1) \
        == N.RMSNORM_EINVAL                                           # tensor scale 0
    assert st(x.data_ptr(), None, None, c.data_ptr(), s.data_ptr(), None, 4, 64, 1e-6, 0.0, float("inf"), 1) \
        == N.RMSNORM_EINVAL
    xf = torch.zeros((4, 64), device=DEV, dtype=torch.float32)
    assert st(xf.data_ptr(), None, None, c.data_ptr(), s.data_ptr(), None, 4, 64, 1e-6, 0.0, 1.0, 0) \
        == N.RMSNORM_EUNSUPPORTED                                     # fp32 I/O
    torch.cuda.synchronize()


@pytest.mark.parametrize("hidden,has_res", [(40960, True), (65536, False), (65536, True)])
def test_nv_long_rows_on_the_bulk_copy_kernel(hidden, has_res):
    """Rows past 32768 elements take the bulk-copy kernel (16 KB pieces) with
    the same NVFP4 epilogue; a grid of 3 blocks over 11 rows as well."""
    wl = W.Workload("nv-long", "bf16", 11, hidden, 1e-5, 1.0, 1.0 if has_res else None, 0.1)
    x, r, w = W.make_inputs(wl, seed=hidden + has_res, device=DEV)
    S = W.NV_TENSOR_SCALE
    p = R.rms_norm_nvfp4_plan_for(x, w=w, residual=r)
    assert p.kernel == N.RMSNORM_KERNEL_TMA and p.chunks_per_thread == 2
    out = R.rms_norm_nvfp4(x, w=w, residual=r, eps=wl.eps, tensor_scale=S)
    torch.cuda.synchronize()
    nv_check(out, x, r, w, wl.eps, S, f"{hidden} library plan")
    q = p.copy()
    q.grid = 3
    out = R.rms_norm_nvfp4(x, w=w, residual=r, eps=wl.eps, tensor_scale=S, plan=q)
    torch.cuda.synchronize()
    nv_check(out, x, r, w, wl.eps, S, f"{hidden} grid 3")
    assert N.rmsnorm_wait_timeouts() == 0
