"""GPU parity of the fused Q+K per-head norm and of the weight-bias form
against the oracle, through the C ABI (GB300 only)."""
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


def qk_oracle(qkv, wl, q_w, k_w, weight_bias=None):
    b = wl.weight_bias if weight_bias is None else weight_bias
    return oracle.rmsnorm_qk(W.to_numpy_bits(qkv), wl.q_heads, wl.k_heads, wl.head_dim,
                             q_w=W.to_numpy_bits(q_w), k_w=W.to_numpy_bits(k_w), eps=wl.eps, dtype=wl.dtype,
                             weight_bias=b, threads=THREADS)


def check_qk(y, qkv_in, wl, q_w, k_w, what, weight_bias=None):
    qy, ky = qk_oracle(qkv_in, wl, q_w, k_w, weight_bias)
    yb = W.to_numpy_bits(y)
    qc, kc = wl.q_heads * wl.head_dim, wl.k_heads * wl.head_dim
    ok, rep = parity.compare_y(yb[:, :qc].reshape(qy.shape), qy, wl.dtype)
    assert ok, f"{what}: query heads {rep}"
    ok, rep = parity.compare_y(yb[:, qc:qc + kc].reshape(ky.shape), ky, wl.dtype)
    assert ok, f"{what}: key heads {rep}"


@pytest.mark.parametrize("name", list(W.QK_WORKLOADS))
def test_qk_workload_out_of_place_and_in_place(name):
    wl = W.QK_WORKLOADS[name]
    qkv, q_w, k_w = W.make_qk_inputs(wl, device=DEV)
    keep = qkv.clone()
    y = R.qk_norm(qkv, wl.q_heads, wl.k_heads, wl.head_dim, q_w, k_w, eps=wl.eps, weight_bias=wl.weight_bias)
    torch.cuda.synchronize()
    assert torch.equal(qkv.view(torch.int16), keep.view(torch.int16)), "input changed"
    check_qk(y, qkv, wl, q_w, k_w, name)
    span = (wl.q_heads + wl.k_heads) * wl.head_dim
    assert torch.equal(y[:, span:].view(torch.int16), keep[:, span:].view(torch.int16)), "value heads changed"
    # in place
    inplace = keep.clone()
    R.qk_norm(inplace, wl.q_heads, wl.k_heads, wl.head_dim, q_w, k_w, eps=wl.eps, weight_bias=wl.weight_bias,
              out=inplace)
    torch.cuda.synchronize()
    assert torch.equal(inplace.view(torch.int16), y.view(torch.int16))


def test_qk_strided_views_and_padding():
    wl = W.QKWorkload("pad", "bf16", 33, 4, 2, 2, 128, 1e-6, 1.0, 0.1)
    # x rows padded to a larger stride; y a view into a wider buffer with its own stride
    qkv, q_w, k_w = W.make_qk_inputs(wl, device=DEV, stride=wl.width + 64)
    ybuf = torch.full((wl.tokens, wl.width + 192), -7.0, device=DEV, dtype=torch.bfloat16)
    y = ybuf[:, 64:64 + wl.width + 64]
    R.qk_norm(qkv, wl.q_heads, wl.k_heads, wl.head_dim, q_w, k_w, eps=wl.eps, out=y)
    torch.cuda.synchronize()
    check_qk(y, qkv, wl, q_w, k_w, "strided")
    span = (wl.q_heads + wl.k_heads) * wl.head_dim
    assert bool((ybuf[:, :64] == -7.0).all()) and bool((ybuf[:, 64 + span:] == -7.0).all())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("head_dim", [64, 128, 256, 127, 8])
@pytest.mark.parametrize("bias", [0.0, 1.0])
def test_qk_every_plan(dtype, head_dim, bias):
    wl = W.QKWorkload("qk-sweep", dtype, 37, 4, 2, 1, head_dim, 1e-5, 1.5, 0.1, weight_bias=bias,
                      w_mean=0.0 if bias else 1.0)
    qkv, q_w, k_w = W.make_qk_inputs(wl, seed=head_dim, device=DEV)
    code = R.dtype_code(qkv.dtype)
    esz = 2 if dtype == "bf16" else 4
    vec_ok = (head_dim * esz) % 16 == 0 and (wl.width * esz) % 16 == 0
    plans = [p for p in all_plans(wl.tokens * 6, head_dim, code, vec_ok)
             if p.kernel == N.RMSNORM_KERNEL_LOOP or p.threads_per_row <= 32]
    assert plans
    qy, ky = qk_oracle(qkv, wl, q_w, k_w)
    for p in plans:
        y = R.qk_norm(qkv, wl.q_heads, wl.k_heads, head_dim, q_w, k_w, eps=wl.eps, weight_bias=bias, plan=p)
        torch.cuda.synchronize()
        yb = W.to_numpy_bits(y)
        qc, kc = wl.q_heads * head_dim, wl.k_heads * head_dim
        ok1, rep1 = parity.compare_y(yb[:, :qc].reshape(qy.shape), qy, dtype)
        ok2, rep2 = parity.compare_y(yb[:, qc:qc + kc].reshape(ky.shape), ky, dtype)
        assert ok1 and ok2, f"plan {p.as_dict()}: {rep1} {rep2}"
        if p.kernel == N.RMSNORM_KERNEL_REG and p.rows_per_block > 1 and head_dim == 128:
            # a block holding one head row (of its rows_per_block slots): same bits
            q = p.copy()
            q.rows_per_block = 1
            q.grid = wl.tokens * 6
            y1 = R.qk_norm(qkv, wl.q_heads, wl.k_heads, head_dim, q_w, k_w, eps=wl.eps, weight_bias=bias, plan=q)
            torch.cuda.synchronize()
            assert parity.bits_equal(W.to_numpy_bits(y1), yb), q.as_dict()
    # the library's own plan
    y = R.qk_norm(qkv, wl.q_heads, wl.k_heads, head_dim, q_w, k_w, eps=wl.eps, weight_bias=bias)
    torch.cuda.synchronize()
    check_qk(y, qkv, wl, q_w, k_w, "default plan")


def test_qk_without_weights_and_one_group():
    for qh, kh in ((3, 0), (0, 5), (2, 2)):
        wl = W.QKWorkload("now", "f32", 19, qh, kh, 1, 64, 1e-6, 1.0, None)
        qkv, _, _ = W.make_qk_inputs(wl, seed=qh * 7 + kh, device=DEV)
        y = R.qk_norm(qkv, qh, kh, 64, eps=wl.eps)
        torch.cuda.synchronize()
        check_qk(y, qkv, wl, None, None, f"no weights q={qh} k={kh}")


def test_qk_matches_contiguous_rows_bitwise():
    """The same head, laid out as a contiguous row, gives the same bits: the
    per-row schedule depends on the row size only."""
    wl = W.QK_WORKLOADS["qk_bf16_64tok_q32_k8_v8_hd128"]
    qkv, _, _ = W.make_qk_inputs(wl, device=DEV)
    y = R.qk_norm(qkv, wl.q_heads, 0, wl.head_dim, eps=wl.eps)
    rows = qkv[:, :wl.q_heads * wl.head_dim].contiguous().view(-1, wl.head_dim)
    yc = R.rms_norm(rows, eps=wl.eps)
    torch.cuda.synchronize()
    assert torch.equal(y[:, :wl.q_heads * wl.head_dim].contiguous().view(-1, wl.head_dim).view(torch.int16),
                       yc.view(torch.int16))


# ------------------------------------------------------------ weight bias

@pytest.mark.parametrize("rows,hidden", [(131, 576), (9, 4096), (33, 1025), (4, 65536), (64, 128)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_weight_bias_every_plan(rows, hidden, dtype):
    wl = W.Workload("wbias", dtype, rows, hidden, 1e-5, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=rows + hidden, device=DEV)
    w = (w.float() - 1.0).to(w.dtype)   # zero-centred weights, as stored for the (1 + w) form
    xn, rn, wn = W.to_numpy_bits(x), W.to_numpy_bits(r), W.to_numpy_bits(w)
    yr, hr, _ = oracle.rmsnorm(xn, w=wn, residual=rn, eps=wl.eps, dtype=dtype, threads=THREADS, weight_bias=1.0)
    code = R.dtype_code(x.dtype)
    esz = 2 if dtype == "bf16" else 4
    plans = [None] + all_plans(rows, hidden, code, (hidden * esz) % 16 == 0, odd_ch=True, tma=True)
    for p in plans:
        y, h = R.rms_norm(x, w=w, residual=r, eps=wl.eps, weight_bias=1.0, plan=p)
        torch.cuda.synchronize()
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
        assert ok, f"plan {None if p is None else p.as_dict()}: {rep}"
        assert parity.bits_equal(W.to_numpy_bits(h), hr)


def test_weight_bias_zero_is_plain_op():
    wl = W.WORKLOADS["bf16_4096x576"]
    x, _, w = W.make_inputs(wl, device=DEV)
    a = R.rms_norm(x, w=w, eps=wl.eps)
    y = torch.empty_like(x)
    N.rmsnorm_fwd_ex(x.data_ptr(), None, w.data_ptr(), y.data_ptr(), None, wl.rows, wl.hidden, wl.eps, 0.0,
                     N.RMSNORM_BF16, None, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), y.view(torch.int16))
