"""The cluster kernel: a row split over the blocks of a thread-block cluster.

Rows past 32 KB with a residual run with one cluster of 2..8 blocks a row,
each block holding a 16 KB slice (32 KB for fp32 rows past 128 KB) in
registers; the blocks' partial sums of squares meet in distributed shared
memory behind one cluster barrier.  Checks, all through the C ABI against
the oracle:
  - every cluster size the planner makes (3 to 8 blocks, ragged last slices,
    both slice sizes) and every weight form (none, w, w + bias, the cast
    order), y within the tolerance and residual_out bit-exact;
  - bits that do not depend on the cluster size (more blocks than the row
    needs), the grid (fewer clusters than rows, striding), or the row count;
  - in-place calls (y over x, residual_out over the residual);
  - the plan the device path makes is the pure host planner's.
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
    from row_reduction_norm_gb300 import _native as N

THREADS = os.cpu_count() or 1
DEV = "cuda"

# (dtype, hidden): the planner's cluster sizes 3..8, ragged and exact last
# slices, 16 KB, 20 KB (rows of 64 to 80 KB) and (fp32 past 128 KB) 32 KB
# slices
SHAPES = [("bf16", 16392), ("bf16", 24576), ("bf16", 32768), ("bf16", 32776), ("bf16", 40960), ("bf16", 40968),
          ("bf16", 57344), ("bf16", 65536),
          ("f32", 8196), ("f32", 20480), ("f32", 32768), ("f32", 32772), ("f32", 40960), ("f32", 65536)]


def _expected(dtype, hidden):
    V = 8 if dtype == "bf16" else 4
    units = hidden // V
    ch = 4 if units <= 8 * 1024 else 8
    if ch == 4 and -(-units // 1024) == 5:   # rows of 64 to 80 KB: four 20 KB slices
        ch = 5
    return ch, -(-units // (256 * ch))


def _oracle(x, r, w, eps, dtype, weight_bias=0.0, cast=False):
    xn, rn, wn = W.to_numpy_bits(x), W.to_numpy_bits(r), W.to_numpy_bits(w)
    if cast:
        y, h, n64 = oracle.rmsnorm_cast(xn, w=wn, residual=rn, eps=eps, dtype=dtype, threads=THREADS)
        return y, h, n64, wn
    y, h, _ = oracle.rmsnorm(xn, w=wn, residual=rn, eps=eps, dtype=dtype, threads=THREADS,
                             weight_bias=weight_bias)
    return y, h, None, wn


def _check(y, h, ref, dtype, cast, what):
    yr, hr, n64, wn = ref
    if cast and dtype == "bf16":
        ok, rep = parity.compare_cast_bf16(W.to_numpy_bits(y), n64, wn, oracle.bf16_from_double)
    else:
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
    assert ok, f"{what}: y differs from the oracle: {rep}"
    assert parity.bits_equal(W.to_numpy_bits(h), hr), f"{what}: residual_out is not bit-exact"


@pytest.mark.parametrize("dtype,hidden", SHAPES)
@pytest.mark.parametrize("form", ["w", "none", "bias", "cast"])
def test_library_plan_matches_oracle(dtype, hidden, form):
    if form == "cast" and dtype != "bf16":
        pytest.skip("the cast order is a bf16 form")
    rows = 5
    has_w = form != "none"
    wl = W.Workload("cluster", dtype, rows, hidden, 1e-6, 1.0, 1.0, 0.1 if has_w else None)
    x, r, w = W.make_inputs(wl, seed=hidden + 7 * len(form), device=DEV)
    p = R.plan_for(x, w=w, residual=r)
    ch, ctas = _expected(dtype, hidden)
    assert (p.kernel, p.regime, p.chunks_per_thread, p.cluster_ctas) == \
        (N.RMSNORM_KERNEL_CLUSTER, N.RMSNORM_REGIME_CLUSTER, ch, ctas), p.as_dict()
    assert p.grid == rows * ctas and p.block_threads == 256
    bias = 1.0 if form == "bias" else 0.0
    y, h = R.rms_norm(x, w=w, residual=r, eps=wl.eps, weight_bias=bias, cast_before_weight=form == "cast")
    torch.cuda.synchronize()
    _check(y, h, _oracle(x, r, w, wl.eps, dtype, bias, form == "cast"), dtype, form == "cast",
           f"{dtype} {hidden} {form}")


@pytest.mark.parametrize("dtype,hidden", [("bf16", 40960), ("bf16", 16392), ("f32", 32772), ("f32", 65536)])
def test_cluster_size_and_grid_change_no_bit(dtype, hidden):
    """Blocks past the row end add +0 to the fixed tree over 8 partial slots,
    and clusters that stride over rows do each row the same way: every such
    plan gives the library plan's bits."""
    rows = 13
    wl = W.Workload("cluster-bits", dtype, rows, hidden, 1e-6, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=hidden + 1, device=DEV)
    p = R.plan_for(x, w=w, residual=r)
    y0, h0 = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    torch.cuda.synchronize()
    _check(y0, h0, _oracle(x, r, w, wl.eps, dtype), dtype, False, "library plan")
    variants = []
    for c in range(p.cluster_ctas, 9):
        for clusters in (rows, 4, 1):
            q = p.copy()
            q.cluster_ctas, q.threads_per_row = c, 256 * c
            q.grid, q.persistent = clusters * c, int(clusters < rows)
            q.pdl = (c + clusters) % 2
            variants.append(q)
    for q in variants:
        y1, h1 = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=q)
        torch.cuda.synchronize()
        assert torch.equal(y1, y0), q.as_dict()
        assert torch.equal(h1, h0), q.as_dict()


def test_fp32_slice_sizes_both_match_oracle():
    """fp32 rows of 128 KB fit eight 16 KB slices or four 32 KB slices: the
    planner takes the first; both match the oracle (their trees differ, so
    their bits may)."""
    rows, hidden = 6, 32768
    wl = W.Workload("cluster-f32", "f32", rows, hidden, 1e-6, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=5, device=DEV)
    ref = _oracle(x, r, w, wl.eps, "f32")
    p = R.plan_for(x, w=w, residual=r)
    assert (p.chunks_per_thread, p.cluster_ctas) == (4, 8)
    q = p.copy()
    q.chunks_per_thread, q.cluster_ctas, q.threads_per_row, q.grid = 8, 4, 1024, rows * 4
    for plan in (p, q):
        y, h = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=plan)
        torch.cuda.synchronize()
        _check(y, h, ref, "f32", False, f"slices of {plan.chunks_per_thread * 4} KB")


@pytest.mark.parametrize("dtype,hidden", [("bf16", 40960), ("f32", 49152)])
def test_batch_invariance(dtype, hidden):
    """A row's bits do not depend on how many rows the launch has."""
    wl = W.Workload("cluster-batch", dtype, 300, hidden, 1e-6, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=9, device=DEV)
    y, h = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    torch.cuda.synchronize()
    for k in (0, 1, 151, 299):
        y1, h1 = R.rms_norm(x[k:k + 1].contiguous(), w=w, residual=r[k:k + 1].contiguous(), eps=wl.eps)
        torch.cuda.synchronize()
        assert torch.equal(y1[0], y[k]) and torch.equal(h1[0], h[k]), k
    g = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 299], g.integers(0, 300, 40)]))
    idx = torch.as_tensor(rows, device=DEV)
    ref = _oracle(x[idx], r[idx], w, wl.eps, dtype)
    _check(y[idx], h[idx], ref, dtype, False, "sampled rows of 300")


@pytest.mark.parametrize("dtype,hidden", [("bf16", 65536), ("f32", 24576)])
def test_in_place(dtype, hidden):
    """y over x and residual_out over the residual: each block reads its
    slice before it writes the same slice, and no block touches another's."""
    wl = W.Workload("cluster-inplace", dtype, 17, hidden, 1e-6, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=11, device=DEV)
    ref = _oracle(x, r, w, wl.eps, dtype)
    assert R.plan_for(x, w=w, residual=r).kernel == N.RMSNORM_KERNEL_CLUSTER
    y, h = R.rms_norm(x, w=w, residual=r, eps=wl.eps, out=x, residual_out=r)
    torch.cuda.synchronize()
    assert y.data_ptr() == x.data_ptr() and h.data_ptr() == r.data_ptr()
    _check(y, h, ref, dtype, False, "in place")


def test_zero_rows_and_device_plan_is_the_host_plan():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for dtype, code, hidden in (("bf16", N.RMSNORM_BF16, 40960), ("f32", N.RMSNORM_F32, 65536),
                                ("bf16", N.RMSNORM_BF16, 16392)):
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        for rows in (1, 1000):
            x = torch.empty((rows, hidden), device=DEV, dtype=tdt)
            ptr = x.data_ptr()
            p = N.rmsnorm_plan_for(ptr, ptr, ptr, ptr, ptr, rows, hidden, code)
            q = N.rmsnorm_plan_ex(rows, hidden, code, True, True, sms, 4)
            assert p.as_dict() == q.as_dict(), (p.as_dict(), q.as_dict())
        # zero rows: a no-op (an empty tensor's data pointer is NULL)
        x = torch.empty((0, hidden), device=DEV, dtype=tdt)
        y, h = R.rms_norm(x, w=None, residual=torch.empty_like(x), eps=1e-6)
        torch.cuda.synchronize()
        assert y.shape == x.shape and h.shape == x.shape


@pytest.mark.parametrize("dtype,hidden", [("bf16", 40960), ("f32", 65536)])
def test_special_values(dtype, hidden):
    """NaN, +-Inf, zero and tiny rows in a cluster's slices (the NaN and Inf
    fall in other blocks than the first): the partial sums carry them across
    the cluster as the oracle's sum does.  A zero residual keeps h = x."""
    tdt = W.TORCH_DTYPE[dtype]
    x = W.random_rows(dtype, 6, hidden, seed=13, device=DEV)
    x[0, hidden // 3] = float("nan")
    x[1, hidden // 2] = float("inf")
    x[2] = 0.0
    x[3, 0] = float("-inf")
    x[3, hidden - 1] = float("inf")
    x[4] = x[4] * 1e-12
    r = torch.zeros_like(x)
    w = torch.ones(hidden, device=DEV, dtype=tdt)
    assert R.plan_for(x, w=w, residual=r).kernel == N.RMSNORM_KERNEL_CLUSTER
    for eps in (1e-5, 0.0):
        y, h = R.rms_norm(x, w=w, residual=r, eps=eps)
        torch.cuda.synchronize()
        yr, hr, _, _ = _oracle(x, r, w, eps, dtype)
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
        assert ok, f"eps={eps}: {rep}"
        # residual_out: NaN where the oracle has NaN (the payload is not part
        # of the op), every other element bit-exact
        hg = h.float().cpu().numpy()
        nan_g = np.isnan(hg)
        nan_o = np.isnan(W.from_numpy_bits(hr, dtype).float().numpy())
        assert (nan_g == nan_o).all()
        keep = ~nan_g
        assert parity.bits_equal(W.to_numpy_bits(h)[keep], hr[keep])
