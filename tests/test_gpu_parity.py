"""Parity of the CUDA path with the oracle, through the C ABI (GB300 only).

Inputs come from the seeded generators in ``row_reduction_norm_gb300.workloads``;
the same tensors go to the CUDA library and, copied to the host, to the
oracle.  Tolerances are in ``parity.py``.  Every workload runs at its full
size in the launch configuration the benchmark uses (the library's own plan);
the largest one is compared on sampled rows that the oracle computes one by
one.  Forced plans cover every regime on every shape they can run.
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


def oracle_run(x, r, w, eps, dtype, rows=None):
    xn = W.to_numpy_bits(x)
    rn = W.to_numpy_bits(r)
    wn = W.to_numpy_bits(w)
    if rows is not None:
        xn = xn[rows]
        rn = None if rn is None else rn[rows]
    y, h, _ = oracle.rmsnorm(xn, w=wn, residual=rn, eps=eps, dtype=dtype, threads=THREADS)
    return y, h


def check(y, h, x, r, w, eps, dtype, rows=None, what=""):
    yr, hr = oracle_run(x, r, w, eps, dtype, rows)
    yg = W.to_numpy_bits(y)
    hg = W.to_numpy_bits(h)
    if rows is not None:
        yg = yg[rows]
        hg = None if hg is None else hg[rows]
    ok, rep = parity.compare_y(yg, yr, dtype)
    assert ok, f"{what}: y differs from the oracle: {rep}"
    if r is not None:
        assert parity.bits_equal(hg, hr), f"{what}: residual_out is not bit-exact"
    return rep


def gpu_inputs(wl, seed=0, rows=None):
    return W.make_inputs(wl, seed=seed, device=DEV, rows=rows)


# ----------------------------------------------------------------- workloads

SMALL = ["f32_64x256", "bf16_4096x576", "bf16_res_16384x2048", "bf16_qk_262144x128",
         "bf16_decode_1x4096", "bf16_decode_8x4096", "bf16_decode_64x4096"]


@pytest.mark.parametrize("name", SMALL)
def test_workload_full_size(name):
    wl = W.WORKLOADS[name]
    x, r, w = gpu_inputs(wl)
    out = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    y, h = out if r is not None else (out, None)
    torch.cuda.synchronize()
    check(y, h, x, r, w, wl.eps, wl.dtype, what=name)


@pytest.mark.parametrize("name", ["bf16_res_65536x8192_w", "bf16_res_65536x8192_nw", "bf16_4096x32768_w",
                                  "bf16_res_4096x40960_w", "bf16_2048x65536_w", "bf16_res_2048x65536_w",
                                  "f32_res_2048x65536_w"])
def test_workload_large_sampled(name):
    wl = W.WORKLOADS[name]
    x, r, w = gpu_inputs(wl)
    out = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    y, h = out if r is not None else (out, None)
    torch.cuda.synchronize()
    g = np.random.default_rng(17)
    n = 509 if wl.hidden <= 8192 else 61
    rows = np.unique(np.concatenate([[0, 1, wl.rows - 1], g.integers(0, wl.rows, n)]))
    idx = torch.as_tensor(rows, device=DEV)
    xs, ys = x[idx], y[idx]
    rs, hs = (None, None) if r is None else (r[idx], h[idx])
    check(ys, hs, xs, rs, w, wl.eps, wl.dtype, what=name)
    if wl.outlier_frac:
        # outliers are present in the sample (0.1% of entries scaled by 100)
        assert float(xs.float().abs().max()) > 50.0
    del x, r, y, h
    torch.cuda.empty_cache()


# ------------------------------------------------------------ forced plans

def all_plans(rows, hidden, dtype_code, vec_ok, sm_count=152, odd_ch=False, tma=False, min_block=256):
    """Every launch plan that is valid for the shape: all REG (threads, chunks)
    pairs that cover the row (chunks 3 and 6 too with ``odd_ch``, compiled for
    contiguous rows), the bulk-copy kernel with both piece sizes that fit
    (``tma``: contiguous RMSNorm rows), the two-pass kernel (vector / scalar,
    each block size that keeps the accuracy bound), each in a full grid and a
    small (persistent) grid.  ``min_block``: the register kernel's smallest
    block (256 for RMSNorm, 128 for LayerNorm)."""
    V = 8 if dtype_code == N.RMSNORM_BF16 else 4
    plans = []
    if vec_ok:
        nch = hidden // V
        for gt in (4, 8, 16, 32, 64, 128, 256, 512):
            for ch in ((1, 2, 3, 4, 6, 8) if odd_ch else (1, 2, 4, 8)):
                if gt * ch * V < hidden:
                    continue
                p = N.Plan()
                p.kernel = N.RMSNORM_KERNEL_REG
                p.threads_per_row = gt
                p.chunks_per_thread = ch
                p.vec_elems = V
                p.block_threads = gt if gt >= min_block else min_block
                p.rows_per_block = p.block_threads // gt
                plans.append(p)
    if vec_ok and tma:
        esz = 16 // V
        for pc in N.TMA_PIECE_CHUNKS:
            if N.tma_rings(hidden * esz, pc, True, True) is None:
                continue   # valid for every residual / weight form the callers run
            p = N.Plan()
            p.kernel = N.RMSNORM_KERNEL_TMA
            p.regime = N.RMSNORM_REGIME_SMEM
            p.threads_per_row = N.TMA_THREADS_PER_ROW
            p.chunks_per_thread = pc
            p.vec_elems = V
            p.block_threads = N.TMA_BLOCK_THREADS
            p.rows_per_block = 1
            plans.append(p)
    for vec in ([True, False] if vec_ok else [False]):
        ve = V if vec else 1
        for blk in (64, 256, 1024):
            if -(-(hidden // ve) // blk) * ve > 64:
                continue
            p = N.Plan()
            p.kernel = N.RMSNORM_KERNEL_LOOP
            p.vec_elems = ve
            p.block_threads = blk
            p.threads_per_row = blk
            p.rows_per_block = 1
            plans.append(p)
    out = []
    for k, p in enumerate(plans):
        row_blocks = -(-rows // p.rows_per_block)
        for grid in sorted({row_blocks, max(1, min(row_blocks, 3))}):
            q = p.copy()
            q.grid = grid
            q.pdl = (k + grid) % 2   # both launch modes across the set
            out.append(q)
    return out


SWEEP = [(131, 576), (64, 256), (37, 128), (9, 4096), (5, 8192), (3, 2048), (2, 16384),
         (7, 64), (19, 8), (2, 32768)]


@pytest.mark.parametrize("rows,hidden", SWEEP)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_every_plan_matches_oracle(rows, hidden, dtype):
    wl = W.Workload("sweep", dtype, rows, hidden, 1e-5, 1.0, 1.0, 0.1)
    x, r, w = gpu_inputs(wl, seed=hidden + rows)
    code = R.dtype_code(x.dtype)
    yr, hr = oracle_run(x, r, w, wl.eps, dtype)
    yr_nr, _ = oracle_run(x, None, None, wl.eps, dtype)
    plans = all_plans(rows, hidden, code, True, odd_ch=True, tma=True)
    assert plans
    for p in plans:
        y, h = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=p)
        y2 = R.rms_norm(x, eps=wl.eps, plan=p)
        torch.cuda.synchronize()
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
        assert ok, f"plan {p.as_dict()}: {rep}"
        assert parity.bits_equal(W.to_numpy_bits(h), hr), f"plan {p.as_dict()}: residual_out"
        ok, rep = parity.compare_y(W.to_numpy_bits(y2), yr_nr, dtype)
        assert ok, f"plan {p.as_dict()} (no residual, no weight): {rep}"


def _fewer_rows(p, rpb, rows, grid=None):
    q = p.copy()
    q.rows_per_block = rpb
    q.grid = grid or -(-rows // rpb)
    q.persistent = int(q.grid < -(-rows // rpb))
    return q


@pytest.mark.parametrize("rows,hidden,dtype", [(9, 4096, "bf16"), (131, 576, "bf16"), (37, 128, "f32"),
                                               (300, 2048, "bf16"), (5, 64, "bf16")])
def test_rows_per_block_changes_no_bit(rows, hidden, dtype):
    """A register-kernel block may hold fewer rows than it has row slots (the
    plan's rows_per_block; planning takes 1 for launches of no more rows than
    SMs): every such plan, full grid or a grid of 3 blocks striding over the
    rows, gives the bits of the plan that fills every slot, with and without
    a residual and a weight."""
    wl = W.Workload("rpb", dtype, rows, hidden, 1e-5, 1.0, 1.0, 0.1)
    x, r, w = gpu_inputs(wl, seed=hidden + 3 * rows)
    code = R.dtype_code(x.dtype)
    yr, hr = oracle_run(x, r, w, wl.eps, dtype)
    full = [p for p in all_plans(rows, hidden, code, True) if p.kernel == N.RMSNORM_KERNEL_REG
            and p.rows_per_block > 1 and p.grid == -(-rows // p.rows_per_block)]
    assert full
    for p in full:
        y0, h0 = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=p)
        n0 = R.rms_norm(x, eps=wl.eps, plan=p)
        torch.cuda.synchronize()
        ok, rep = parity.compare_y(W.to_numpy_bits(y0), yr, dtype)
        assert ok, f"plan {p.as_dict()}: {rep}"
        for rpb in sorted({1, p.rows_per_block // 2 + 1, p.rows_per_block - 1} - {0, p.rows_per_block}):
            for grid in (None, 3):
                q = _fewer_rows(p, rpb, rows, grid)
                y1, h1 = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=q)
                n1 = R.rms_norm(x, eps=wl.eps, plan=q)
                torch.cuda.synchronize()
                assert parity.bits_equal(W.to_numpy_bits(y1), W.to_numpy_bits(y0)), q.as_dict()
                assert parity.bits_equal(W.to_numpy_bits(h1), hr), q.as_dict()
                assert parity.bits_equal(W.to_numpy_bits(n1), W.to_numpy_bits(n0)), q.as_dict()


def test_decode_launches_spread_rows():
    """Decode batches hold one warp of rows a block (one row for rows of a
    warp or more, 32 / threads_per_row below) while that needs no more blocks
    than SMs; a longer batch fills every slot."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for hidden, per_warp in ((576, 1), (4096, 1), (128, 8), (256, 4)):
        x = torch.empty((1, hidden), device=DEV, dtype=torch.bfloat16)
        for rows in (1, 8, 64, sms):
            p = N.rmsnorm_plan_for(x.data_ptr(), None, x.data_ptr(), x.data_ptr(), None, rows, hidden,
                                   N.RMSNORM_BF16)
            assert p.rows_per_block == min(per_warp, p.block_threads // p.threads_per_row), p.as_dict()
            assert p.grid == -(-rows // p.rows_per_block), p.as_dict()
        p = N.rmsnorm_plan_for(x.data_ptr(), None, x.data_ptr(), x.data_ptr(), None, 40 * sms, hidden,
                               N.RMSNORM_BF16)
        assert p.rows_per_block == p.block_threads // p.threads_per_row


# ------------------------------------------------------------ shape sweep

HIDDENS = [1, 7, 8, 31, 33, 64, 127, 128, 576, 1000, 1024, 1025, 2048, 4096, 8192, 12288,
           16384, 32768, 65536]


@pytest.mark.parametrize("hidden", HIDDENS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_tail_sweep(hidden, dtype):
    for rows in (1, 3, 131):
        for has_res, has_w in ((False, False), (False, True), (True, True), (True, False)):
            if hidden >= 16384 and rows == 131 and (has_res or not has_w):
                continue  # keep the case small; the full option matrix runs at rows 1 and 3
            wl = W.Workload("tail", dtype, rows, hidden, 1e-6, 1.0, 1.0 if has_res else None,
                            0.1 if has_w else None)
            x, r, w = gpu_inputs(wl, seed=rows * 7 + hidden)
            out = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
            y, h = out if r is not None else (out, None)
            torch.cuda.synchronize()
            check(y, h, x, r, w, wl.eps, dtype, what=f"H={hidden} rows={rows} res={has_res} w={has_w}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_regime_query_matches_the_plan(dtype):
    """rmsnorm_regime names the regime of the plan rmsnorm_fwd uses (aligned
    tensors, a weight, no residual) on every width of the tail sweep and on
    row counts from one row to many waves."""
    code = N.RMSNORM_BF16 if dtype == "bf16" else N.RMSNORM_F32
    esz = 2 if dtype == "bf16" else 4
    for hidden in HIDDENS:
        if (hidden * esz) % 16:
            continue
        x = torch.empty((1, hidden), device=DEV, dtype=W.TORCH_DTYPE[dtype])
        for rows in (0, 1, 3, 131, 65536, 1 << 22):
            p = N.rmsnorm_plan_for(x.data_ptr(), None, x.data_ptr(), x.data_ptr(), None, rows, hidden, code)
            assert R.rmsnorm_regime(rows, hidden, code) == p.regime, (hidden, rows, p.as_dict())
    assert N.rmsnorm_regime_status(4, 1 << 17, code) == N.RMSNORM_EUNSUPPORTED


def test_rows_zero_is_noop():
    x = torch.empty((0, 576), device=DEV, dtype=torch.bfloat16)
    y = R.rms_norm(x)
    assert y.shape == (0, 576)


# ------------------------------------------------------ alignment, aliasing

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,hidden", [(33, 2048), (5, 65536), (9, 40960)])
def test_misaligned_base_pointer(dtype, rows, hidden):
    tdt = W.TORCH_DTYPE[dtype]
    buf = W.random_rows(dtype, 1, rows * hidden + 1, seed=4, device=DEV).reshape(-1)
    x = buf[1:].view(rows, hidden)           # one element past a 16-byte boundary
    w = (1 + 0.1 * W.random_rows(dtype, 1, hidden + 1, seed=5, device=DEV)).to(tdt).reshape(-1)[1:]
    ybuf = torch.empty(rows * hidden + 1, device=DEV, dtype=tdt)
    y = ybuf[1:].view(rows, hidden)
    p = R.plan_for(x, w=w, out=y)
    assert p.vec_elems == 1 and p.kernel == N.RMSNORM_KERNEL_LOOP
    R.rms_norm(x, w=w, eps=1e-6, out=y)
    torch.cuda.synchronize()
    check(y, None, x, None, w, 1e-6, dtype, what="misaligned")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("hidden", [576, 2048, 1025])
def test_in_place(dtype, hidden):
    rows = 77
    wl = W.Workload("inplace", dtype, rows, hidden, 1e-5, 1.0, 1.0, 0.1)
    x, r, w = gpu_inputs(wl, seed=8)
    yref, href = oracle_run(x, r, w, wl.eps, dtype)
    yref0, _ = oracle_run(x, None, w, wl.eps, dtype)
    # y written over x, no residual
    xa = x.clone()
    R.rms_norm(xa, w=w, eps=wl.eps, out=xa)
    # residual_out written over residual, y over x
    xb, rb = x.clone(), r.clone()
    R.rms_norm(xb, w=w, residual=rb, eps=wl.eps, out=xb, residual_out=rb)
    # residual_out written over x
    xc, rc = x.clone(), r.clone()
    yc = torch.empty_like(x)
    R.rms_norm(xc, w=w, residual=rc, eps=wl.eps, out=yc, residual_out=xc)
    torch.cuda.synchronize()
    assert parity.compare_y(W.to_numpy_bits(xa), yref0, dtype)[0]
    assert parity.compare_y(W.to_numpy_bits(xb), yref, dtype)[0]
    assert parity.bits_equal(W.to_numpy_bits(rb), href)
    assert parity.compare_y(W.to_numpy_bits(yc), yref, dtype)[0]
    assert parity.bits_equal(W.to_numpy_bits(xc), href)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("hidden", [128, 576, 4096, 1025, 65536])
def test_guard_bands_untouched(dtype, hidden):
    rows = 5
    guard = 4096 // (2 if dtype == "bf16" else 4)
    tdt = W.TORCH_DTYPE[dtype]
    wl = W.Workload("guard", dtype, rows, hidden, 1e-6, 1.0, 1.0, 0.1)
    x, r, w = gpu_inputs(wl, seed=9)
    sentinel = torch.full((rows * hidden + 2 * guard,), -123.0, device=DEV, dtype=tdt)
    ybuf, hbuf = sentinel.clone(), sentinel.clone()
    y = ybuf[guard:guard + rows * hidden].view(rows, hidden)
    h = hbuf[guard:guard + rows * hidden].view(rows, hidden)
    R.rms_norm(x, w=w, residual=r, eps=wl.eps, out=y, residual_out=h)
    torch.cuda.synchronize()
    for buf in (ybuf, hbuf):
        assert bool((buf[:guard] == -123.0).all()) and bool((buf[guard + rows * hidden:] == -123.0).all())
    check(y, h, x, r, w, wl.eps, dtype, what="guard")


# ------------------------------------------------- determinism, invariance

@pytest.mark.parametrize("name", ["bf16_4096x576", "bf16_res_16384x2048", "bf16_qk_262144x128",
                                  "f32_64x256"])
def test_deterministic_and_batch_invariant(name):
    wl = W.WORKLOADS[name]
    x, r, w = gpu_inputs(wl, seed=2)
    a = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    b = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    ya = a[0] if r is not None else a
    yb = b[0] if r is not None else b
    torch.cuda.synchronize()
    assert torch.equal(ya.view(torch.int16) if ya.dtype == torch.bfloat16 else ya.view(torch.int32),
                       yb.view(torch.int16) if yb.dtype == torch.bfloat16 else yb.view(torch.int32))
    # a row normalised alone, or in a short batch, gives the same bits as in the full batch
    for lo, hi in ((0, 1), (5, 13), (wl.rows - 3, wl.rows)):
        part = R.rms_norm(x[lo:hi].contiguous(), w=w,
                          residual=None if r is None else r[lo:hi].contiguous(), eps=wl.eps)
        yp = part[0] if r is not None else part
        torch.cuda.synchronize()
        assert parity.bits_equal(W.to_numpy_bits(yp), W.to_numpy_bits(ya[lo:hi]))


@pytest.mark.parametrize("hidden,has_res", [(576, False), (576, True), (5120, False), (12288, True)])
def test_batch_invariant_across_chunk_fit(hidden, has_res):
    """A launch of many waves takes the chunk count that fits the row exactly
    (3 or 6), a short one of rows wider than a warp the power of two (rows of
    a warp or less take the exact fit in every launch); a row's bits are the
    same in all of them."""
    rows = max(40000 * 576 // hidden, 2000)
    wl = W.Workload("fit", "bf16", rows, hidden, 1e-6, 1.0, 1.0 if has_res else None, 0.1)
    x, r, w = gpu_inputs(wl, seed=hidden + has_res)
    p_big = R.plan_for(x, w=w, residual=r)
    p_small = R.plan_for(x[:13], w=w, residual=None if r is None else r[:13])
    assert p_big.threads_per_row == p_small.threads_per_row
    assert p_big.chunks_per_thread in (3, 6)
    if p_small.threads_per_row > 32:
        assert p_small.chunks_per_thread in (4, 8)
    else:
        # the power-of-two count, forced, gives the same bits as the exact fit
        assert p_small.chunks_per_thread in (3, 6)
        q = p_small.copy()
        q.chunks_per_thread = 4 if p_small.chunks_per_thread == 3 else 8
        forced = R.rms_norm(x[:13].contiguous(), w=w, residual=None if r is None else r[:13].contiguous(),
                            eps=wl.eps, plan=q)
        lib = R.rms_norm(x[:13].contiguous(), w=w, residual=None if r is None else r[:13].contiguous(), eps=wl.eps)
        torch.cuda.synchronize()
        yf = forced[0] if r is not None else forced
        yl = lib[0] if r is not None else lib
        assert parity.bits_equal(W.to_numpy_bits(yf), W.to_numpy_bits(yl))
    out = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    y = out[0] if r is not None else out
    part = R.rms_norm(x[:13].contiguous(), w=w, residual=None if r is None else r[:13].contiguous(), eps=wl.eps)
    yp = part[0] if r is not None else part
    torch.cuda.synchronize()
    assert parity.bits_equal(W.to_numpy_bits(yp), W.to_numpy_bits(y[:13]))
    check(y[:64], None if r is None else out[1][:64], x[:64], None if r is None else r[:64], w, wl.eps, "bf16",
          what=f"H={hidden} res={has_res}")


# ------------------------------------------------------------ special values

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("hidden", [64, 576, 4096, 1025])
def test_special_values(dtype, hidden):
    tdt = W.TORCH_DTYPE[dtype]
    x = W.random_rows(dtype, 6, hidden, seed=12, device=DEV)
    x[0, hidden // 3] = float("nan")
    x[1, hidden // 2] = float("inf")
    x[2] = 0.0
    x[3, 0] = float("-inf")
    x[4] = x[4] * 1e-12       # tiny row: eps dominates (squares stay in the fp32 normal range)
    w = torch.ones(hidden, device=DEV, dtype=tdt)
    for eps in (1e-5, 0.0):
        y = R.rms_norm(x, w=w, eps=eps)
        torch.cuda.synchronize()
        yr, _ = oracle_run(x, None, w, eps, dtype)
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
        assert ok, f"eps={eps}: {rep}"


# ---------------------------------------------------------------- streams

def test_runs_on_the_given_stream():
    wl = W.WORKLOADS["bf16_4096x576"]
    x, r, w = gpu_inputs(wl, seed=1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = R.rms_norm(x, w=w, eps=wl.eps)
    s.synchronize()
    check(y, None, x, None, w, wl.eps, "bf16", what="side stream")


# ------------------------------------------------------------ status codes

def test_status_codes_on_device():
    x = torch.zeros((4, 64), device=DEV, dtype=torch.bfloat16)
    y = torch.empty_like(x)
    p, q = x.data_ptr(), y.data_ptr()
    assert N.rmsnorm_fwd_status(p, None, None, q, None, 4, 64, 1e-6, 1, 0) == N.RMSNORM_OK
    assert N.rmsnorm_fwd_status(p, None, None, q, None, 4, 64, -1.0, 1, 0) == N.RMSNORM_EINVAL
    assert N.rmsnorm_fwd_status(p, None, None, q, None, 4, 64, float("nan"), 1, 0) == N.RMSNORM_EINVAL
    assert N.rmsnorm_fwd_status(p, p, None, q, None, 4, 64, 1e-6, 1, 0) == N.RMSNORM_EINVAL
    assert N.rmsnorm_fwd_status(p, None, None, q, None, 4, 1 << 17, 1e-6, 1, 0) == N.RMSNORM_EUNSUPPORTED
    assert N.rmsnorm_fwd_status(p + 1, None, None, q, None, 4, 8, 1e-6, 1, 0) == N.RMSNORM_EINVAL
    bad = R.rmsnorm_plan(4, 64, 1, True, 152, 1)
    bad.threads_per_row = 3
    assert N.rmsnorm_fwd_plan_status(p, None, None, q, None, 4, 64, 1e-6, 1, bad, 0) == N.RMSNORM_EINVAL
    small = R.rmsnorm_plan(4, 64, 1, True, 152, 1)
    small.chunks_per_thread = 1
    small.threads_per_row = 4
    small.block_threads = 256
    small.rows_per_block = 64
    assert N.rmsnorm_fwd_plan_status(p, None, None, q, None, 4, 64, 1e-6, 1, small, 0) == N.RMSNORM_EINVAL
    torch.cuda.synchronize()


# ------------------------------------------------------ 64-bit addressing

@pytest.mark.parametrize("hidden,rows,has_res,kind", [
    (8192, 288000, False, "reg"),      # x 4.4 GiB: register kernel
    (40960, 57600, False, "tma"),      # x 4.4 GiB: bulk-copy kernel
    (65536, 36000, True, "cluster"),   # x and residual 4.4 GiB each: a cluster of blocks a row
    (65536, 36000, True, "loop"),      # the same, the two-pass kernel forced
])
def test_offsets_past_4gib(hidden, rows, has_res, kind):
    """Tensors larger than 4 GiB: rows near the end sit at byte offsets past
    2^32, checked against the oracle on sampled rows (first, last, and rows
    either side of the 2^31 and 2^32 byte boundaries)."""
    wl = W.Workload("big", "bf16", rows, hidden, 1e-6, 1.0, 1.0 if has_res else None, 0.1)
    x, r, w = gpu_inputs(wl, seed=hidden)
    p = R.plan_for(x, w=w, residual=r)
    if kind == "loop":
        p.kernel, p.regime, p.threads_per_row, p.chunks_per_thread = (N.RMSNORM_KERNEL_LOOP,
                                                                      N.RMSNORM_REGIME_LOOPED, 1024, 0)
        p.block_threads, p.rows_per_block, p.grid, p.persistent, p.cluster_ctas = 1024, 1, rows, 0, 0
    assert p.as_dict()["kernel_name"] == kind
    out = R.rms_norm(x, w=w, residual=r, eps=wl.eps, plan=p)
    y, h = out if r is not None else (out, None)
    torch.cuda.synchronize()
    row_bytes = hidden * 2
    picks = {0, rows - 1}
    for edge in (1 << 31, 1 << 32):
        k = edge // row_bytes
        picks.update({k - 1, k, k + 1})
    idx = torch.as_tensor(sorted(i for i in picks if 0 <= i < rows), device=DEV)
    check(y[idx], None if h is None else h[idx], x[idx], None if r is None else r[idx], w, wl.eps, "bf16",
          what=f"{kind} {rows}x{hidden}")
    del x, r, y, h, out
    torch.cuda.empty_cache()


def test_golden_closed_forms_through_the_kernel():
    # the hand-derived cases of tests/golden/closed_forms.txt through the C ABI,
    # against their exactly rounded values (the usual tolerance; residual_out exact)
    import exact
    import pins
    for c in pins.parse_golden():
        dt = c["dtype"]
        n = len(c["x"])
        enc = lambda vals: pins.to_array([pins.encode_exact(v, dt) for v in vals], dt)

        def dev(a, shape):
            t = torch.from_numpy(a.reshape(shape).copy())
            return (t.view(torch.bfloat16) if dt == "bf16" else t).to(DEV)

        x = dev(enc(c["x"]), (1, n))
        w = None if c["w"] is None else dev(enc(c["w"]), (n,))
        r = None if c["residual"] is None else dev(enc(c["residual"]), (1, n))
        out = R.rms_norm(x, w=w, residual=r, eps=float(c["eps"]))
        y, h = out if r is not None else (out, None)
        torch.cuda.synchronize()
        want = pins.to_array([exact.round_sqrt(s, q, dt) for s, q in zip(c["sign"], c["y2"])], dt).reshape(1, n)
        ok, rep = parity.compare_y(W.to_numpy_bits(y), want, dt)
        assert ok, f"{c['name']}: {rep}"
        if c.get("resout") is not None:
            assert np.array_equal(W.to_numpy_bits(h), enc(c["resout"]).reshape(1, n)), c["name"]
