"""The host-buffer call ``rmsnorm_fwd_host`` (GB300 only).

Rows in host memory go through the device in chunks: uploads, one
``rmsnorm_fwd`` launch a chunk, read-backs, on three streams over two halves
of the caller's workspace.  Checks, against the oracle and against
``rmsnorm_fwd`` on device copies of the same rows (bit for bit: the schedule
does not depend on the row count):
  - ragged last chunks, one chunk, a chunk per row, every kernel family's
    widths (warp, CTA, cluster with a residual, bulk copy without one);
  - pinned and pageable host memory;
  - back-to-back calls sharing one workspace (a later call's uploads wait for
    the earlier call's read-backs of the same half), on a side stream, with
    the results read after that stream alone is synchronised;
  - argument errors.
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


def _host(t, pinned):
    h = t.cpu()
    return h.pin_memory() if pinned else h


def _check(y, h, x, r, w, eps, dtype, what):
    yr, hr, _ = oracle.rmsnorm(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r), eps=eps,
                               dtype=dtype, threads=THREADS)
    ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
    assert ok, f"{what}: y differs from the oracle: {rep}"
    if r is not None:
        assert parity.bits_equal(W.to_numpy_bits(h), hr), f"{what}: residual_out is not bit-exact"


CASES = [
    # dtype, rows, hidden, residual, weight, chunk_rows
    ("bf16", 1001, 4096, True, True, 128),     # 8 chunks, the last ragged
    ("bf16", 300, 576, False, True, 300),      # one chunk
    ("bf16", 37, 2048, True, False, 1),        # a chunk a row
    ("f32", 513, 1024, True, True, 64),
    ("bf16", 40, 40960, True, True, 16),       # cluster kernel
    ("bf16", 24, 40960, False, True, 7),       # bulk-copy kernel
    ("f32", 9, 65536, True, True, 4),          # cluster kernel, 32 KB slices
    ("bf16", 5, 130, True, True, 2),           # rows not a multiple of 16 bytes: scalar kernel
]


@pytest.mark.parametrize("dtype,rows,hidden,has_res,has_w,chunk", CASES)
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_call_matches_oracle_and_device_call(dtype, rows, hidden, has_res, has_w, chunk, pinned):
    wl = W.Workload("host", dtype, rows, hidden, 1e-6, 1.0, 1.0 if has_res else None, 0.1 if has_w else None)
    x, r, w = W.make_inputs(wl, seed=rows + hidden, device=DEV)
    hx, hr, hw = _host(x, pinned), None if r is None else _host(r, pinned), None if w is None else _host(w, pinned)
    hy = torch.empty_like(hx).pin_memory() if pinned else torch.empty_like(hx)
    hh = None if r is None else (torch.empty_like(hx).pin_memory() if pinned else torch.empty_like(hx))
    s = torch.cuda.Stream()
    out = R.rms_norm_host(hx, w=hw, residual=hr, eps=wl.eps, out=hy, residual_out=hh, chunk_rows=chunk, stream=s)
    s.synchronize()
    y, h = out if r is not None else (out, None)
    assert y.data_ptr() == hy.data_ptr()
    _check(y, h, x, r, w, wl.eps, dtype, f"{dtype} {rows}x{hidden} chunk {chunk}")
    dev = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    torch.cuda.synchronize()
    yd, hd = dev if r is not None else (dev, None)
    assert torch.equal(y, yd.cpu()), "the host call's y is not rmsnorm_fwd's"
    if r is not None:
        assert torch.equal(h, hd.cpu())


def test_back_to_back_calls_share_a_workspace():
    """Three calls on one workspace and one side stream, inputs changing each
    time: every later call's uploads wait until the earlier call's
    read-backs of the same half are done."""
    wl = W.Workload("host-seq", "bf16", 700, 8192, 1e-6, 1.0, 1.0, 0.1)
    chunk = 64
    need = R.rmsnorm_host_workspace_bytes(chunk, wl.hidden, N.RMSNORM_BF16, True)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    runs = []
    for k in range(3):
        x, r, w = W.make_inputs(wl, seed=50 + k, device=DEV)
        hx, hr, hw = x.cpu().pin_memory(), r.cpu().pin_memory(), w.cpu().pin_memory()
        hy, hh = torch.empty_like(hx).pin_memory(), torch.empty_like(hx).pin_memory()
        R.rms_norm_host(hx, w=hw, residual=hr, eps=wl.eps, out=hy, residual_out=hh, chunk_rows=chunk,
                        workspace=ws, stream=s)
        runs.append((x, r, w, hy, hh))
    s.synchronize()
    for k, (x, r, w, hy, hh) in enumerate(runs):
        _check(hy, hh, x, r, w, wl.eps, "bf16", f"call {k}")


def test_zero_rows_and_bad_arguments():
    x = torch.zeros((0, 256), dtype=torch.bfloat16)
    y = R.rms_norm_host(x)
    torch.cuda.synchronize()
    assert y.shape == x.shape
    xs = torch.zeros((8, 256), dtype=torch.bfloat16).pin_memory()
    small = torch.empty(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError):
        R.rms_norm_host(xs, workspace=small)
    with pytest.raises(ValueError):
        R.rms_norm_host(xs.to(DEV))
    need = R.rmsnorm_host_workspace_bytes(4, 256, N.RMSNORM_BF16, False)
    ws = torch.empty(need + 256, dtype=torch.uint8, device=DEV)
    ys = torch.empty_like(xs).pin_memory()
    st = N.rmsnorm_fwd_host_status(xs.data_ptr(), None, None, ys.data_ptr(), None, 8, 256, 1e-6,
                                   N.RMSNORM_BF16, ws.data_ptr() + 16, need, 4, 0)
    assert st == N.RMSNORM_EINVAL                     # workspace not on a 256-byte boundary
    st = N.rmsnorm_fwd_host_status(xs.data_ptr(), None, None, ys.data_ptr(), None, 8, 256, 1e-6,
                                   N.RMSNORM_BF16, ws.data_ptr(), need, 4, 0)
    torch.cuda.synchronize()
    assert st == N.RMSNORM_OK
    assert bool((ys.float() == 0).all())              # zero rows normalise to zeros
