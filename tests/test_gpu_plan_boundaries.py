"""Every planner boundary on GB300: the widths where the kernel family
changes, one 16-byte unit either side, both dtypes, with and without a
residual, against the oracle.

Boundaries (bytes a row): 16 KB (256 threads x 4 chunks to x 8), 32 KB
(register kernel to the cluster kernel with a residual, to the bulk-copy
kernel without), 80 KB (bulk copy: weight resident to weight from L2),
128 KB (cluster: 16 KB to 32 KB fp32 slices), 192 KB (bulk copy to the
two-pass kernel without a residual).  The family each width plans is
asserted too, so a boundary that moved shows up here.
"""
import os

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


def _family(row_bytes, dtype, has_res):
    """The kernel family the planner takes for aligned rows (the rule the
    header states)."""
    if row_bytes <= 32 * 1024:
        return "reg"
    if has_res:
        return "cluster"
    return "tma" if row_bytes <= 192 * 1024 else "loop"


def _widths(dtype):
    esz = 2 if dtype == "bf16" else 4
    V = 16 // esz
    out = set()
    for kb in (16, 32, 80, 128, 192):
        h = kb * 1024 // esz
        out.update({h - V, h, h + V})
    return sorted(w for w in out if 0 < w <= 65536)


CASES = [(d, h) for d in ("bf16", "f32") for h in _widths(d)]


@pytest.mark.parametrize("dtype,hidden", CASES)
@pytest.mark.parametrize("has_res", [False, True], ids=["plain", "residual"])
def test_boundary_width(dtype, hidden, has_res):
    esz = 2 if dtype == "bf16" else 4
    rows = 3
    wl = W.Workload("boundary", dtype, rows, hidden, 1e-6, 1.0, 1.0 if has_res else None, 0.1)
    x, r, w = W.make_inputs(wl, seed=hidden * 2 + has_res, device=DEV)
    p = R.plan_for(x, w=w, residual=r)
    assert p.as_dict()["kernel_name"] == _family(hidden * esz, dtype, has_res), p.as_dict()
    out = R.rms_norm(x, w=w, residual=r, eps=wl.eps)
    y, h = out if r is not None else (out, None)
    torch.cuda.synchronize()
    yr, hr, _ = oracle.rmsnorm(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r), eps=wl.eps,
                               dtype=dtype, threads=THREADS)
    ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, dtype)
    assert ok, f"{dtype} {hidden} res={has_res} ({p.as_dict()['kernel_name']}): {rep}"
    if r is not None:
        assert parity.bits_equal(W.to_numpy_bits(h), hr)
    # the cast order and the weight bias take the same family
    if dtype == "bf16":
        yc, _ = (R.rms_norm(x, w=w, residual=r, eps=wl.eps, cast_before_weight=True) if has_res
                 else (R.rms_norm(x, w=w, eps=wl.eps, cast_before_weight=True), None))
        torch.cuda.synchronize()
        yrc, _, n64 = oracle.rmsnorm_cast(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r),
                                          eps=wl.eps, dtype=dtype, threads=THREADS)
        ok, rep = parity.compare_cast_bf16(W.to_numpy_bits(yc), n64, W.to_numpy_bits(w), oracle.bf16_from_double)
        assert ok, f"cast order {hidden} res={has_res}: {rep}"
    yb = R.rms_norm(x, w=w, residual=r, eps=wl.eps, weight_bias=1.0)
    yb = yb[0] if r is not None else yb
    torch.cuda.synchronize()
    ybr, _, _ = oracle.rmsnorm(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r), eps=wl.eps,
                               dtype=dtype, threads=THREADS, weight_bias=1.0)
    ok, rep = parity.compare_y(W.to_numpy_bits(yb), ybr, dtype)
    assert ok, f"weight bias {hidden} res={has_res}: {rep}"
