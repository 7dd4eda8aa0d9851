"""GPU parity of RMSNorm with MXFP8 output against the oracle, through the
C ABI (GB300 only).  Codes and scales are integers decided by floating
point: they must equal the oracle's except where the exact value lies within
the fp32 error of a decision boundary (``parity.compare_mx``)."""
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


def mx_check(out, x, r, w, eps, dtype, what, weight_bias=0.0):
    codes, scales = out[0], out[1]
    co, so, ho, v64 = oracle.rmsnorm_mxfp8(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r),
                                           eps=eps, dtype=dtype, weight_bias=weight_bias, threads=THREADS)
    ok, rep = parity.compare_mx(codes.cpu().numpy(), scales.cpu().numpy(), co, so, v64, oracle.e4m3_from_double)
    assert ok, f"{what}: {rep}"
    if r is not None:
        assert parity.bits_equal(W.to_numpy_bits(out[2]), ho), f"{what}: residual_out"
    return rep


@pytest.mark.parametrize("name", ["bf16_4096x576", "bf16_res_16384x2048", "bf16_qk_262144x128", "f32_64x256"])
def test_mx_workloads(name):
    wl = W.WORKLOADS[name]
    x, r, w = W.make_inputs(wl, device=DEV)
    out = R.rms_norm_mxfp8(x, w=w, residual=r, eps=wl.eps)
    torch.cuda.synchronize()
    rep = mx_check(out, x, r, w, wl.eps, wl.dtype, name)
    assert rep["code_flips"] <= 1e-4 * x.numel()


@pytest.mark.parametrize("rows,hidden", [(37, 576), (9, 4096), (64, 128), (3, 32), (5, 2048), (2, 16384)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_mx_every_plan(rows, hidden, dtype):
    wl = W.Workload("mx-sweep", dtype, rows, hidden, 1e-5, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=rows + hidden, device=DEV)
    code = R.dtype_code(x.dtype)
    lpb = 4 if dtype == "bf16" else 8
    plans = [p for p in all_plans(rows, hidden, code, True)
             if p.kernel == N.RMSNORM_KERNEL_REG and p.threads_per_row >= lpb]
    assert plans
    for p in plans:
        for ww, rr, b in ((w, r, 0.0), (None, None, 0.0), (w, None, 1.0)):
            out = R.rms_norm_mxfp8(x, w=ww, residual=rr, eps=wl.eps, weight_bias=b, plan=p)
            torch.cuda.synchronize()
            mx_check(out, x, rr, ww, wl.eps, dtype, f"plan {p.as_dict()} w={ww is not None} res={rr is not None}",
                     weight_bias=b)
        if p.rows_per_block > 1 and p.grid == -(-rows // p.rows_per_block):
            # one row a block: the same codes and scales
            q = p.copy()
            q.rows_per_block, q.grid = 1, rows
            a = R.rms_norm_mxfp8(x, w=w, residual=r, eps=wl.eps, plan=p)
            c = R.rms_norm_mxfp8(x, w=w, residual=r, eps=wl.eps, plan=q)
            torch.cuda.synchronize()
            assert all(torch.equal(u, v) for u, v in zip(a, c)), q.as_dict()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_mx_special_blocks_and_dynamic_range(dtype):
    tdt = W.TORCH_DTYPE[dtype]
    x = W.random_rows(dtype, 6, 256, seed=8, device=DEV)
    x[0, 5] = float("nan")                 # block 0 of row 0 is NaN; the rest of row 0 is NaN too (NaN row)
    x[1, 40] = float("inf")
    x[2] = 0.0                             # zero row, eps > 0: all-zero blocks (scale code 0)
    x[3, :32] = x[3, :32] * 1e-6           # a tiny block beside normal ones
    x[4, 64:96] = x[4, 64:96] * 1e3        # an outlier block
    out = R.rms_norm_mxfp8(x, eps=1e-5)
    torch.cuda.synchronize()
    mx_check(out, x, None, None, 1e-5, dtype, "special")
    codes, scales = out
    assert int(scales[2, 0]) == 0 and int(codes[2].abs().max()) == 0


def test_mx_argument_checks():
    x = torch.zeros((4, 64), device=DEV, dtype=torch.bfloat16)
    c = torch.empty((4, 64), device=DEV, dtype=torch.uint8)
    s = torch.empty((4, 2), device=DEV, dtype=torch.uint8)
    ok = N.rmsnorm_fwd_mxfp8_status(x.data_ptr(), None, None, c.data_ptr(), s.data_ptr(), None, 4, 64, 1e-6, 0.0, 1)
    assert ok == N.RMSNORM_OK
    assert N.rmsnorm_fwd_mxfp8_status(x.data_ptr(), None, None, c.data_ptr(), s.data_ptr(), None, 4, 48, 1e-6, 0.0,
                                      1) == N.RMSNORM_EINVAL          # hidden not a multiple of 32
    assert N.rmsnorm_fwd_mxfp8_status(x.data_ptr(), None, None, c.data_ptr() + 8, s.data_ptr(), None, 4, 64, 1e-6,
                                      0.0, 1) == N.RMSNORM_EINVAL     # codes not 16-byte aligned
    assert N.rmsnorm_fwd_mxfp8_status(x.data_ptr(), None, None, c.data_ptr(), None, None, 4, 64, 1e-6, 0.0, 1) \
        == N.RMSNORM_EINVAL                                           # no scales
    # fp32 rows of 65536 (256 KB) fit neither registers nor the bulk-copy
    # kernel's rings: refused at planning, before any launch
    big = N.rmsnorm_fwd_mxfp8_status(x.data_ptr(), None, None, c.data_ptr(), s.data_ptr(), None, 1, 65536, 1e-6,
                                     0.0, 0)
    assert big == N.RMSNORM_EUNSUPPORTED
    torch.cuda.synchronize()


def test_mx_matches_plain_op_dequantised():
    """Dequantised codes are within half an E4M3 step of the plain op's fp32-accurate values."""
    wl = W.WORKLOADS["bf16_res_16384x2048"]
    x, r, w = W.make_inputs(wl, rows=256, device=DEV)
    codes, scales, _ = R.rms_norm_mxfp8(x, w=w, residual=r, eps=wl.eps)
    torch.cuda.synchronize()
    _, _, _, v64 = oracle.rmsnorm_mxfp8(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r),
                                        eps=wl.eps, dtype="bf16", threads=THREADS)
    vals = parity._e4m3_values(codes.cpu().numpy()).reshape(256, -1, 32)
    sc = np.ldexp(1.0, scales.cpu().numpy().astype(np.int64) - 127)[:, :, None]
    deq = (vals * sc).reshape(256, -1)
    step = np.ldexp(1.0, np.frexp(np.abs(v64) + 1e-300)[1] - 4)       # E4M3 quantum of |v|
    floor_q = np.ldexp(1.0, scales.cpu().numpy().astype(np.int64) - 127 - 9)[:, :, None]
    limit = np.maximum(step, np.broadcast_to(floor_q, (256, 2048 // 32, 32)).reshape(256, -1)) * 0.5 * (1 + 4e-6)
    scale_full = np.broadcast_to(sc, (256, 2048 // 32, 32)).reshape(256, -1)
    in_range = np.abs(v64) <= 448.0 * scale_full          # saturated values (448..512 x scale) excluded
    assert np.all((np.abs(deq - v64) <= limit) | ~in_range)
    assert np.all(np.abs(deq[~in_range]) == 448.0 * scale_full[~in_range])


@pytest.mark.parametrize("dtype,hidden,has_res,has_w", [("bf16", 40960, True, True), ("bf16", 65536, False, True),
                                                        ("bf16", 65536, True, True), ("f32", 24576, True, True),
                                                        ("f32", 40960, True, True)])
def test_mx_long_rows_on_the_bulk_copy_kernel(dtype, hidden, has_res, has_w):
    """Rows too long for registers take the bulk-copy kernel (16 KB pieces)
    with the same block-scaled epilogue; a grid of 3 blocks over 11 rows also
    checks that blocks walk several rows."""
    wl = W.Workload("mx-long", dtype, 11, hidden, 1e-5, 1.0, 1.0 if has_res else None, 0.1 if has_w else None)
    x, r, w = W.make_inputs(wl, seed=hidden + has_res, device=DEV)
    p = R.rms_norm_mxfp8_plan_for(x, w=w, residual=r)
    assert p.kernel == N.RMSNORM_KERNEL_TMA and p.chunks_per_thread == 2
    out = R.rms_norm_mxfp8(x, w=w, residual=r, eps=wl.eps)
    torch.cuda.synchronize()
    mx_check(out, x, r, w, wl.eps, dtype, f"{dtype} {hidden} library plan")
    q = p.copy()
    q.grid = 3
    out = R.rms_norm_mxfp8(x, w=w, residual=r, eps=wl.eps, weight_bias=1.0 if has_w else 0.0, plan=q)
    torch.cuda.synchronize()
    mx_check(out, x, r, w, wl.eps, dtype, f"{dtype} {hidden} grid 3", weight_bias=1.0 if has_w else 0.0)
    assert N.rmsnorm_wait_timeouts() == 0
