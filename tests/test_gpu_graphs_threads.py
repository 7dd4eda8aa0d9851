"""The C ABI under CUDA graph capture and under concurrent host threads
(GB300 only): launches recorded in a graph replay with new inputs; calls from
several host threads, each on its own stream, give the oracle's results."""
import os
import threading

import pytest
import torch

import oracle
import parity
from row_reduction_norm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import row_reduction_norm_gb300 as R

THREADS = os.cpu_count() or 1
DEV = "cuda"


def _ref(x, r, w, eps, dtype):
    y, h, _ = oracle.rmsnorm(W.to_numpy_bits(x), w=W.to_numpy_bits(w), residual=W.to_numpy_bits(r), eps=eps,
                             dtype=dtype, threads=THREADS)
    return y, h


def test_graph_capture_and_replay_with_new_inputs():
    wl = W.WORKLOADS["bf16_res_16384x2048"]
    x, r, w = W.make_inputs(wl, rows=512, device=DEV)
    y = torch.empty_like(x)
    h = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        R.rms_norm(x, w=w, residual=r, eps=wl.eps, out=y, residual_out=h)   # fills the per-device caches
        ln_y = R.layer_norm(x, w=w, eps=1e-5)
        qkv = torch.empty((64, 48 * 128), device=DEV, dtype=torch.bfloat16).normal_()
        R.qk_norm(qkv, 32, 8, 128, eps=1e-6, out=qkv)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        R.rms_norm(x, w=w, residual=r, eps=wl.eps, out=y, residual_out=h)
        R.layer_norm(x, w=w, eps=1e-5, out=ln_y)
    for seed in (11, 12):
        x2, r2, _ = W.make_inputs(wl, seed=seed, rows=512, device=DEV)
        x.copy_(x2)
        r.copy_(r2)
        g.replay()
        torch.cuda.synchronize()
        yr, hr = _ref(x, r, w, wl.eps, "bf16")
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, "bf16")
        assert ok, rep
        assert parity.bits_equal(W.to_numpy_bits(h), hr)
        direct = R.layer_norm(x, w=w, eps=1e-5)
        torch.cuda.synchronize()
        assert torch.equal(direct.view(torch.int16), ln_y.view(torch.int16))


def test_concurrent_host_threads_on_own_streams():
    wl = W.WORKLOADS["bf16_4096x576"]
    n_threads, iters = 4, 20
    inputs = [W.make_inputs(wl, seed=100 + k, device=DEV) for k in range(n_threads)]
    outs = [torch.empty_like(inputs[k][0]) for k in range(n_threads)]
    errors = []

    def work(k):
        try:
            s = torch.cuda.Stream()
            x, _, w = inputs[k]
            with torch.cuda.stream(s):
                for _ in range(iters):
                    R.rms_norm(x, w=w, eps=wl.eps, out=outs[k])
            s.synchronize()
        except Exception as ex:   # reported below
            errors.append(repr(ex))

    ts = [threading.Thread(target=work, args=(k,)) for k in range(n_threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    for k in range(n_threads):
        x, _, w = inputs[k]
        yr, _ = _ref(x, None, w, wl.eps, "bf16")
        ok, rep = parity.compare_y(W.to_numpy_bits(outs[k]), yr, "bf16")
        assert ok, rep


@pytest.mark.parametrize("has_res", [False, True], ids=["bulk-copy", "cluster"])
def test_long_row_kernels_in_a_graph_and_from_threads(has_res):
    """The kernels of rows past 32 KB -- the shared-memory (bulk copy) kernel
    without a residual, a thread-block cluster a row with one -- recorded in a
    CUDA graph and replayed on new inputs, and launched from several host
    threads at once, each on its own stream; no bounded wait runs out."""
    from row_reduction_norm_gb300 import _native as N
    wl = W.Workload("graph_long", "bf16", 40, 40960, 1e-6, 1.0, 1.0 if has_res else None, 0.1)
    x, r, w = W.make_inputs(wl, seed=3, device=DEV)
    y = torch.empty_like(x)
    h = torch.empty_like(x) if has_res else None
    want = N.RMSNORM_KERNEL_CLUSTER if has_res else N.RMSNORM_KERNEL_TMA
    assert R.plan_for(x, w=w, residual=r).kernel == want
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        R.rms_norm(x, w=w, residual=r, eps=wl.eps, out=y, residual_out=h)   # fills the per-device caches
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        R.rms_norm(x, w=w, residual=r, eps=wl.eps, out=y, residual_out=h)
    for seed in (21, 22):
        x2, r2, _ = W.make_inputs(wl, seed=seed, device=DEV)
        x.copy_(x2)
        if has_res:
            r.copy_(r2)
        g.replay()
        torch.cuda.synchronize()
        yr, hr = _ref(x, r, w, wl.eps, "bf16")
        ok, rep = parity.compare_y(W.to_numpy_bits(y), yr, "bf16")
        assert ok, rep
        if has_res:
            assert parity.bits_equal(W.to_numpy_bits(h), hr)

    n_threads = 3
    inputs = [W.make_inputs(wl, seed=200 + k, device=DEV) for k in range(n_threads)]
    outs = [(torch.empty_like(i[0]), torch.empty_like(i[0]) if has_res else None) for i in inputs]
    errors = []

    def work(k):
        try:
            st = torch.cuda.Stream()
            xk, rk, wk = inputs[k]
            with torch.cuda.stream(st):
                for _ in range(10):
                    R.rms_norm(xk, w=wk, residual=rk, eps=wl.eps, out=outs[k][0], residual_out=outs[k][1])
            st.synchronize()
        except Exception as ex:   # reported below
            errors.append(repr(ex))

    ts = [threading.Thread(target=work, args=(k,)) for k in range(n_threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    for k in range(n_threads):
        xk, rk, wk = inputs[k]
        yr, hr = _ref(xk, rk, wk, wl.eps, "bf16")
        ok, rep = parity.compare_y(W.to_numpy_bits(outs[k][0]), yr, "bf16")
        assert ok, rep
        if has_res:
            assert parity.bits_equal(W.to_numpy_bits(outs[k][1]), hr)
    torch.cuda.synchronize()
    assert N.rmsnorm_wait_timeouts() == 0
