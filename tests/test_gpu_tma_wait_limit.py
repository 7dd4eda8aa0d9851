"""The bulk-copy kernel's bounded waits running out, on purpose, on a GB300.

Every wait of the kernel (for a copy to land, for a ring slot to free) has a
time limit; a block whose wait runs out finishes without valid output, waits
for its copies in flight and adds 1 to the counter ``rmsnorm_wait_timeouts``
reads.  The C ABI's test hook ``rmsnorm_tma_wait_test`` shortens the limit
to a millisecond and makes the first consumer warp of block 0 keep one x
slot, so that block's producer waits for a slot that never frees.  Nothing
faults and no wait is unbounded.  The checks: the counter rises by exactly
one, the other blocks' rows are right, a launch with the short limit and no
withheld slot is right and counts nothing, and the next ordinary launch is
right.  This file sorts after every test that expects the counter at zero.
"""
import os
import time

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
LIMIT_NS = 1_000_000   # 1 ms


def _oracle(x, r, w, eps):
    y, h, _ = oracle.rmsnorm(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r), eps=eps,
                             dtype="bf16", threads=THREADS)
    return y, h


def _hook(x, r, w, y, h, plan, withhold, eps, limit=LIMIT_NS):
    s = torch.cuda.current_stream()
    return N.rmsnorm_tma_wait_test_status(x.data_ptr(), None if r is None else r.data_ptr(), w.data_ptr(),
                                          y.data_ptr(), None if h is None else h.data_ptr(), x.shape[0], x.shape[1],
                                          eps, N.RMSNORM_BF16, plan, limit, withhold, s.cuda_stream)


@pytest.mark.parametrize("has_res,hidden", [(False, 40960), (True, 40960), (False, 49152)],
                         ids=["plain", "residual", "weight-from-L2"])
def test_withheld_slot_times_out_and_the_next_launch_is_right(has_res, hidden):
    rows, grid = 12, 3
    wl = W.Workload("wait", "bf16", rows, hidden, 1e-6, 1.0, 1.0 if has_res else None, 0.1)
    x, r, w = W.make_inputs(wl, seed=21, device=DEV)
    y = torch.empty_like(x)
    h = torch.empty_like(x) if has_res else None
    # the bulk-copy plan of these rows without a residual (with one, the
    # library plans a cluster of blocks a row); with the residual it runs with
    # 16 KB pieces, the weight resident
    plan = R.plan_for(x, w=w, out=y)
    assert plan.kernel == N.RMSNORM_KERNEL_TMA
    if has_res:
        plan.chunks_per_thread = 2
        assert N.tma_rings(hidden * 2, 2, True, True)[2] > 0
    plan.grid, plan.persistent = grid, 1          # block 0 walks rows 0, 3, 6, 9
    yr, hr = _oracle(x, r, w, wl.eps)
    torch.cuda.synchronize()
    n0 = N.rmsnorm_wait_timeouts()

    # the short limit alone never fires on a launch that runs normally
    assert _hook(x, r, w, y, h, plan, 0, wl.eps) == N.RMSNORM_OK
    torch.cuda.synchronize()
    assert N.rmsnorm_wait_timeouts() == n0
    ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, "bf16")
    assert ok, rep

    # block 0 keeps one slot: its waits run out, it counts itself once
    y.fill_(0)
    t0 = time.time()
    assert _hook(x, r, w, y, h, plan, 1, wl.eps) == N.RMSNORM_OK
    torch.cuda.synchronize()
    took = time.time() - t0
    assert N.rmsnorm_wait_timeouts() == n0 + 1
    assert took < 5.0, f"the failed launch took {took:.3f} s"
    others = [i for i in range(rows) if i % grid != 0]
    ok, rep = parity.compare_y(W.to_numpy_bits(y)[others], yr[others], "bf16")
    assert ok, f"rows of the blocks that did not give up: {rep}"
    if has_res:
        assert parity.bits_equal(W.to_numpy_bits(h)[others], hr[others])

    # the context is fine and the next ordinary launches are right
    for _ in range(2):
        y.fill_(0)
        out = R.rms_norm(x, w=w, residual=r, eps=wl.eps, out=y, residual_out=h, plan=plan)
        torch.cuda.synchronize()
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, "bf16")
        assert ok, rep
        if has_res:
            assert parity.bits_equal(W.to_numpy_bits(out[1]), hr)
    assert N.rmsnorm_wait_timeouts() == n0 + 1


def test_hook_rejects_bad_arguments():
    x = torch.zeros((2, 40960), device=DEV, dtype=torch.bfloat16)
    w = torch.ones(40960, device=DEV, dtype=torch.bfloat16)
    y = torch.empty_like(x)
    plan = R.plan_for(x, w=w, out=y)
    reg = R.plan_for(x[:, :1024].contiguous(), w=w[:1024].contiguous())
    assert _hook(x, None, w, y, None, reg, 0, 1e-6) == N.RMSNORM_EINVAL        # not a bulk-copy plan
    assert _hook(x, None, w, y, None, plan, 2, 1e-6) == N.RMSNORM_EINVAL       # withhold is 0 or 1
    assert _hook(x, None, w, y, None, plan, 0, 1e-6, limit=2_000_000_000) == N.RMSNORM_EINVAL   # above 1 s
    assert _hook(x, None, w, y, None, plan, 0, -1.0) == N.RMSNORM_EINVAL       # the op's own checks
    torch.cuda.synchronize()
