"""The bulk-copy (TMA) kernel: rows staged in a shared-memory ring.

Three kinds of check, all through the C ABI:
  - long rows (past the register capacity) against the oracle, every
    weight / residual form, both piece sizes, grids smaller than the row count
    so each block walks many rows and the ring wraps many times;
  - bit equality with the register kernel at 512 threads a row on rows both
    kernels can take (same per-thread order and tree, so the same bits);
  - the bounded-wait counter stays at zero.
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


def tma_plan(pc, grid, V):
    p = N.Plan()
    p.kernel = N.RMSNORM_KERNEL_TMA
    p.regime = N.RMSNORM_REGIME_SMEM
    p.threads_per_row = N.TMA_THREADS_PER_ROW
    p.chunks_per_thread = pc
    p.vec_elems = V
    p.block_threads = N.TMA_BLOCK_THREADS
    p.rows_per_block = 1
    p.grid = grid
    p.pdl = 1
    return p


def reg512_plan(hidden, V, rows):
    p = N.Plan()
    p.kernel = N.RMSNORM_KERNEL_REG
    p.threads_per_row = 512
    need = -(-(hidden // V) // 512)
    ch = 1
    while ch < need:
        ch *= 2
    p.chunks_per_thread = ch
    p.vec_elems = V
    p.block_threads = 512
    p.rows_per_block = 1
    p.grid = rows
    p.pdl = 1
    return p


def fits(hidden, esz, pc, res=True, w=True):
    return N.tma_rings(hidden * esz, pc, res, w) is not None


def oracle_ref(x, r, w, eps, dtype, weight_bias=0.0):
    y, h, _ = oracle.rmsnorm(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r), eps=eps,
                             dtype=dtype, threads=THREADS, weight_bias=weight_bias)
    return y, h


# rows the library plans on the bulk-copy kernel without a residual (32 to 80
# KB; with a residual it plans the cluster kernel), and longer rows it can run
# when forced (up to 160 KB with a residual and a weight)
PLANNED = [("bf16", 32776), ("bf16", 40000), ("bf16", 40960), ("f32", 16388), ("f32", 20480)]
LONG = PLANNED + [("bf16", 65536), ("f32", 24576), ("f32", 40960)]


@pytest.mark.parametrize("dtype,hidden", PLANNED)
def test_long_rows_library_plan(dtype, hidden):
    esz = 2 if dtype == "bf16" else 4
    for rows, has_res, has_w in ((1, False, False), (7, True, True), (40, True, False), (19, False, True)):
        wl = W.Workload("long", dtype, rows, hidden, 1e-6, 1.0, 1.0 if has_res else None,
                        0.1 if has_w else None)
        x, r, w = W.make_inputs(wl, seed=hidden + rows, device=DEV)
        p = R.plan_for(x, w=w, residual=r)
        if has_res:
            assert p.kernel == N.RMSNORM_KERNEL_CLUSTER and p.regime == N.RMSNORM_REGIME_CLUSTER
            p = R.plan_for(x, w=w)          # the bulk-copy plan, forced with the residual
            p.chunks_per_thread = 2
        assert p.kernel == N.RMSNORM_KERNEL_TMA and p.regime == N.RMSNORM_REGIME_SMEM
        assert p.chunks_per_thread == (4 if dtype == "bf16" and not has_res else 2)
        assert fits(hidden, esz, p.chunks_per_thread, has_res, has_w)
        out = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=p)
        y, h = out if r is not None else (out, None)
        torch.cuda.synchronize()
        yr, hr = oracle_ref(x, r, w, wl.eps, dtype)
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
        assert ok, f"rows={rows} res={has_res} w={has_w}: {rep}"
        if r is not None:
            assert parity.bits_equal(W.to_numpy_bits(h), hr)


@pytest.mark.parametrize("dtype,hidden", [("bf16", 65536), ("f32", 24576), ("f32", 49152)])
def test_rows_past_80kb_plan_by_residual(dtype, hidden):
    """Past 80 KB the weight cannot stay resident beside the row: without a
    residual the library plans the bulk-copy kernel with 32 KB pieces (the
    weight read from L2), with a residual the cluster kernel; both match the
    oracle."""
    for has_res in (False, True):
        wl = W.Workload("past80", dtype, 9, hidden, 1e-6, 1.0, 1.0 if has_res else None, 0.1)
        x, r, w = W.make_inputs(wl, seed=hidden + has_res, device=DEV)
        p = R.plan_for(x, w=w, residual=r)
        if has_res:
            assert p.kernel == N.RMSNORM_KERNEL_CLUSTER
        else:
            assert p.kernel == N.RMSNORM_KERNEL_TMA and p.chunks_per_thread == 4
        out = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
        y, h = out if r is not None else (out, None)
        torch.cuda.synchronize()
        yr, hr = oracle_ref(x, r, w, wl.eps, dtype)
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
        assert ok, f"res={has_res}: {rep}"
        if r is not None:
            assert parity.bits_equal(W.to_numpy_bits(h), hr)


@pytest.mark.parametrize("dtype,hidden", LONG)
@pytest.mark.parametrize("pc", [1, 2, 4])
def test_long_rows_ring_wraps(dtype, hidden, pc):
    """Grids of 1, 3 and 7 blocks over 29 rows: a block walks up to 29 rows,
    so every slot is refilled many times and both barrier parities recur."""
    esz = 2 if dtype == "bf16" else 4
    if not fits(hidden, esz, pc):
        pytest.skip("row larger than the ring at this piece size")
    wl = W.Workload("wrap", dtype, 29, hidden, 1e-5, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=pc * 1000 + hidden, device=DEV)
    yr, hr = oracle_ref(x, r, w, wl.eps, dtype, weight_bias=1.0)
    for grid in (1, 3, 7):
        y, h = R.rms_norm(x, w=w, residual=r, eps=wl.eps, weight_bias=1.0, plan=tma_plan(pc, grid, 16 // esz))
        torch.cuda.synchronize()
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
        assert ok, f"grid={grid}: {rep}"
        assert parity.bits_equal(W.to_numpy_bits(h), hr), f"grid={grid}: residual_out"


SAME = [("bf16", 576), ("bf16", 4096), ("bf16", 8192), ("bf16", 12296), ("bf16", 32768),
        ("f32", 4096), ("f32", 8200), ("f32", 16384)]


@pytest.mark.parametrize("dtype,hidden", SAME)
def test_same_bits_as_register_kernel(dtype, hidden):
    V = 8 if dtype == "bf16" else 4
    esz = 16 // V
    rows = 37
    for has_res, has_w in ((True, True), (False, False), (False, True)):
        wl = W.Workload("same", dtype, rows, hidden, 1e-6, 1.0, 1.0 if has_res else None,
                        0.1 if has_w else None)
        x, r, w = W.make_inputs(wl, seed=hidden * 3 + has_res, device=DEV)
        ref = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=reg512_plan(hidden, V, rows))
        yref, href = ref if r is not None else (ref, None)
        for pc in (1, 2, 4):
            if not fits(hidden, esz, pc, has_res, has_w):
                continue
            for grid in (rows, 5):
                p = tma_plan(pc, grid, V)
                out = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=p)
                y, h = out if r is not None else (out, None)
                torch.cuda.synchronize()
                assert parity.bits_equal(W.to_numpy_bits(y), W.to_numpy_bits(yref)), \
                    f"pc={pc} grid={grid} res={has_res} w={has_w}"
                if r is not None:
                    assert parity.bits_equal(W.to_numpy_bits(h), W.to_numpy_bits(href))


@pytest.mark.parametrize("dtype,hidden", [("bf16", 40000), ("f32", 24576)])
def test_long_rows_special_values_and_in_place(dtype, hidden):
    tdt = W.TORCH_DTYPE[dtype]
    x = W.random_rows(dtype, 5, hidden, seed=31, device=DEV)
    x[0, hidden // 3] = float("nan")
    x[1, hidden - 1] = float("inf")
    x[2] = 0.0
    x[3] = x[3] * 1e-12
    w = (1 + 0.1 * W.random_rows(dtype, 1, hidden, seed=32, device=DEV)).to(tdt).reshape(-1)
    for eps in (1e-5, 0.0):
        yr, _ = oracle_ref(x, None, w, eps, dtype)
        y = R.rms_norm(x, w=w, eps=eps)
        xi = x.clone()
        R.rms_norm(xi, w=w, eps=eps, out=xi)      # y written over x
        torch.cuda.synchronize()
        for got in (y, xi):
            ok, rep = parity.compare_y(W.to_numpy_bits(got), yr, dtype)
            assert ok, f"eps={eps}: {rep}"


def test_long_rows_full_size_sampled():
    """2048 rows of 65536 bf16 with a residual and a weight (256 MB a tensor):
    the library plan, compared on sampled rows."""
    wl = W.Workload("long_full", "bf16", 2048, 65536, 1e-6, 1.0, 1.0, 0.1)
    x, r, w = W.make_inputs(wl, seed=5, device=DEV)
    y, h = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 151, 152, 2047], np.random.default_rng(3).integers(0, 2048, 60)]))
    idx = torch.as_tensor(rows, device=DEV)
    yr, hr = oracle_ref(x[idx], r[idx], w, wl.eps, "bf16")
    ok, rep = parity.compare_y(W.to_numpy_bits(y[idx]), yr, "bf16")
    assert ok, rep
    assert parity.bits_equal(W.to_numpy_bits(h[idx]), hr)
    del x, r, y, h
    torch.cuda.empty_cache()


def test_no_wait_ran_out():
    torch.cuda.synchronize()
    assert N.rmsnorm_wait_timeouts() == 0
