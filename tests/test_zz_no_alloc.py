"""rmsnorm_fwd_host_static: the host-buffer call on the library's own device
scratch (a file-scope __device__ array), against rmsnorm_fwd_host with a
caller workspace, on two calls (GB300 only).  Collected last.

Both calls must give the same bits (each chunk is one rmsnorm_fwd launch and
the schedule does not depend on the row count), and the second call, after
the first has brought the scratch in, must leave the device's free memory
unchanged: the entry point allocates nothing.
"""
import pytest
import torch

from row_reduction_norm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import row_reduction_norm_gb300 as R
    from row_reduction_norm_gb300 import _native as N

DEV = "cuda"


def _pinned(t):
    return None if t is None else t.cpu().pin_memory()


@pytest.mark.parametrize("dtype,rows,hidden,has_res", [("bf16", 3000, 8192, True), ("f32", 40, 65536, False)])
def test_static_scratch_call_matches_the_workspace_call(dtype, rows, hidden, has_res):
    wl = W.Workload("noalloc", dtype, rows, hidden, 1e-6, 1.0, 1.0 if has_res else None, 0.1)
    x, r, w = W.make_inputs(wl, seed=rows, device=DEV)
    hx, hr, hw = _pinned(x), _pinned(r), _pinned(w)
    code = R.dtype_code(x.dtype)
    ptr = lambda t: None if t is None else t.data_ptr()
    y_ref = R.rms_norm_host(hx, w=hw, residual=hr, eps=wl.eps, chunk_rows=97)
    torch.cuda.synchronize()
    y_ref, h_ref = y_ref if has_res else (y_ref, None)
    for call in range(2):
        hy = torch.empty_like(hx).pin_memory()
        hh = torch.empty_like(hx).pin_memory() if has_res else None
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        s = torch.cuda.current_stream()
        N.rmsnorm_fwd_host_static(ptr(hx), ptr(hr), ptr(hw), ptr(hy), ptr(hh), rows, hidden, wl.eps, code,
                                  s.cuda_stream)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert torch.equal(hy, y_ref), f"call {call}: y differs from rmsnorm_fwd_host's"
        if has_res:
            assert torch.equal(hh, h_ref), f"call {call}: residual_out differs"
        if call == 1:
            assert free1 == free0, "the call changed the device's free memory"
