"""Dependent chains of launches under programmatic dependent launch (GB300 only).

Every library launch carries the programmatic-stream-serialisation attribute,
so launch k+1 may start while launch k drains; its blocks execute
``griddepcontrol.wait`` before they read an input.  These tests make launch
k+1 read what launch k wrote -- y becomes the next x, residual_out the next
residual -- in place and out of place, eagerly and inside a captured CUDA
graph, on every kernel family (register warp / CTA, two-pass vector and
scalar, shared-memory rings fed by bulk copies, a row split over the blocks
of a thread-block cluster, and a chain that switches family every launch),
and compare every step with the oracle applied to the previous step's output
as the GPU wrote it.

In-place chains keep a snapshot per step: launch "snap" normalises buffer A
into B[k] (out of place), then launch "in place" normalises A over itself
with the same plan.  Both compute the same bits from the same input, so
B[k] is what A holds after step k; B[k+1] is then checked against the oracle
of B[k], and the final A against the last snapshot, bit for bit.  A read that
overtook the previous launch's writes (or a write that overtook its reads)
shows up as a mismatch.
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
    from test_gpu_parity import all_plans

THREADS = os.cpu_count() or 1
DEV = "cuda"
STEPS = 6


def _bits(t):
    return W.to_numpy_bits(t)


def _plans(family, rows, hidden, dtype, x, w, r):
    """The launch plans one chain cycles through (one per step, repeating)."""
    code = N.RMSNORM_BF16 if dtype == "bf16" else N.RMSNORM_F32
    lib = R.plan_for(x, w=w, residual=r, out=torch.empty_like(x), residual_out=None if r is None else
                     torch.empty_like(x))
    if family in ("tma", "long"):
        # past 32 KB: a cluster of blocks a row with a residual; the bulk-copy
        # kernel without one (past 80 KB with the weight read from L2)
        want = N.RMSNORM_REGIME_CLUSTER if r is not None else N.RMSNORM_REGIME_SMEM
        assert lib.regime == want, lib.as_dict()
        return [lib]
    if family in ("warp", "cta"):
        want = {"warp": N.RMSNORM_REGIME_WARP, "cta": N.RMSNORM_REGIME_CTA}[family]
        assert lib.regime == want, lib.as_dict()
        if rows <= torch.cuda.get_device_properties(0).multi_processor_count:
            assert lib.rows_per_block == 1, lib.as_dict()   # the decode spread
        return [lib]
    forced = all_plans(rows, hidden, code, True, odd_ch=True, tma=True)
    full_grid = [p for p in forced if p.grid == -(-rows // p.rows_per_block)]
    for p in full_grid:
        p.pdl = 1
    loop_vec = [p for p in full_grid if p.kernel == N.RMSNORM_KERNEL_LOOP and p.vec_elems != 1]
    loop_scalar = [p for p in full_grid if p.kernel == N.RMSNORM_KERNEL_LOOP and p.vec_elems == 1]
    if family == "loop":
        return [loop_vec[0], loop_scalar[0]]
    assert family == "mixed"
    tma = [p for p in full_grid if p.kernel == N.RMSNORM_KERNEL_TMA]
    reg = [p for p in full_grid if p.kernel == N.RMSNORM_KERNEL_REG and p.threads_per_row == 512]
    persistent = lib.copy()
    persistent.grid = min(persistent.grid, 5)   # blocks stride over the rows
    persistent.persistent = 1
    chain = [lib, tma[0], loop_vec[-1], reg[0], loop_scalar[0], persistent, tma[-1]]
    if r is not None:
        # the cluster kernel on a row one 16 KB slice covers: two blocks a
        # cluster (the second past the row end), then three clusters striding
        # over the rows
        V = 8 if dtype == "bf16" else 4
        cl = R.rmsnorm_plan_ex(rows, 40960, code, True, True, 152, 4)
        cl.cluster_ctas, cl.threads_per_row = 2, 512
        cl.chunks_per_thread = 4
        assert 2 * 256 * 4 * V >= hidden
        cl.grid = rows * 2
        few = cl.copy()
        few.grid, few.persistent = 6, 1
        chain[2:2] = [cl]
        chain.append(few)
    return chain


CASES = [
    # family, dtype, rows, hidden
    ("warp", "bf16", 8192, 576),
    ("cta", "bf16", 2048, 4096),
    ("cta", "f32", 1024, 2048),
    ("cta", "bf16", 64, 4096),      # a decode batch: one row a block
    ("warp", "bf16", 100, 576),     # the same, rows of a warp
    ("tma", "bf16", 300, 40960),
    ("long", "bf16", 200, 49152),
    ("loop", "bf16", 1000, 4096),
    ("mixed", "bf16", 1000, 8192),
]


def _check_step(y, h, x_bits, r_bits, w_bits, eps, dtype, what):
    yr, hr, _ = oracle.rmsnorm(x_bits, w=w_bits, residual=r_bits, eps=eps, dtype=dtype, threads=THREADS)
    ok, rep = parity.compare_y(_bits(y), yr, dtype)
    assert ok, f"{what}: y differs from the oracle: {rep}"
    if r_bits is not None:
        assert parity.bits_equal(_bits(h), hr), f"{what}: residual_out is not bit-exact"


def _run(issue, graph, reset):
    """Issue the chain on a side stream, eagerly or as a captured graph.  The
    graph form runs the chain once eagerly first (the library fills its
    per-device caches outside any capture), then resets the inputs, captures
    and replays it."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        issue()
    s.synchronize()
    if not graph:
        return
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        issue()
    reset()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("has_res", [False, True], ids=["plain", "residual"])
@pytest.mark.parametrize("family,dtype,rows,hidden", CASES)
def test_chain_out_of_place(family, dtype, rows, hidden, has_res, graph):
    wl = W.Workload("chain", dtype, rows, hidden, 1e-6, 1.0, 1.0 if has_res else None, 0.1)
    x0, r0, w = W.make_inputs(wl, seed=rows + hidden, device=DEV)
    X = [x0.clone()] + [torch.empty_like(x0) for _ in range(STEPS)]
    H = [r0.clone() if has_res else None] + [torch.empty_like(x0) if has_res else None for _ in range(STEPS)]
    plans = _plans(family, rows, hidden, dtype, x0, w, r0)

    def issue():
        for k in range(1, STEPS + 1):
            R.rms_norm(X[k - 1], w=w, residual=H[k - 1], eps=wl.eps, out=X[k], residual_out=H[k],
                       plan=plans[(k - 1) % len(plans)])

    def reset():
        for t in X[1:] + [h for h in H[1:] if h is not None]:
            t.fill_(0)

    _run(issue, graph, reset)
    wn = _bits(w)
    for k in range(1, STEPS + 1):
        _check_step(X[k], H[k], _bits(X[k - 1]), None if not has_res else _bits(H[k - 1]), wn, wl.eps, dtype,
                    f"{family} step {k} plan {plans[(k - 1) % len(plans)].as_dict()}")


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("has_res", [False, True], ids=["plain", "residual"])
@pytest.mark.parametrize("family,dtype,rows,hidden", CASES)
def test_chain_in_place(family, dtype, rows, hidden, has_res, graph):
    wl = W.Workload("chain", dtype, rows, hidden, 1e-6, 1.0, 1.0 if has_res else None, 0.1)
    x0, r0, w = W.make_inputs(wl, seed=3 * rows + hidden, device=DEV)
    A = x0.clone()
    Ra = r0.clone() if has_res else None
    B = [torch.empty_like(x0) for _ in range(STEPS)]
    HB = [torch.empty_like(x0) if has_res else None for _ in range(STEPS)]
    plans = _plans(family, rows, hidden, dtype, x0, w, r0)

    def issue():
        for k in range(STEPS):
            p = plans[k % len(plans)]
            R.rms_norm(A, w=w, residual=Ra, eps=wl.eps, out=B[k], residual_out=HB[k], plan=p)   # snapshot
            R.rms_norm(A, w=w, residual=Ra, eps=wl.eps, out=A, residual_out=Ra, plan=p)        # in place

    def reset():
        A.copy_(x0)
        if has_res:
            Ra.copy_(r0)
        for t in B + [h for h in HB if h is not None]:
            t.fill_(0)

    _run(issue, graph, reset)
    wn = _bits(w)
    prev_x, prev_r = _bits(x0), _bits(r0) if has_res else None
    for k in range(STEPS):
        _check_step(B[k], HB[k], prev_x, prev_r, wn, wl.eps, dtype,
                    f"{family} in place, step {k} plan {plans[k % len(plans)].as_dict()}")
        prev_x, prev_r = _bits(B[k]), _bits(HB[k]) if has_res else None
    assert np.array_equal(_bits(A), prev_x), "the in-place result differs from its out-of-place twin"
    if has_res:
        assert np.array_equal(_bits(Ra), prev_r), "the in-place residual_out differs from its twin"


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("rows,hidden,forced", [(4096, 768, None), (512, 4096, "loop")])
def test_layernorm_chain(rows, hidden, forced, graph):
    """LayerNorm launches chained the same way (register and three-pass kernels)."""
    wl = W.Workload("ln-chain", "bf16", rows, hidden, 1e-5, 1.0, 1.0, 0.1, b_std=0.1, x_mean=0.25)
    x0, r0, w, b = W.make_ln_inputs(wl, seed=rows, device=DEV)
    X = [x0.clone()] + [torch.empty_like(x0) for _ in range(STEPS)]
    H = [r0.clone()] + [torch.empty_like(x0) for _ in range(STEPS)]
    plan = None
    if forced:
        plan = [p for p in all_plans(rows, hidden, N.RMSNORM_BF16, True, odd_ch=True, min_block=128)
                if p.kernel == N.RMSNORM_KERNEL_LOOP and p.grid == rows][0]
        plan.pdl = 1

    def issue():
        for k in range(1, STEPS + 1):
            R.layer_norm(X[k - 1], w=w, b=b, residual=H[k - 1], eps=wl.eps, out=X[k], residual_out=H[k],
                         plan=plan)

    def reset():
        for t in X[1:] + H[1:]:
            t.fill_(0)

    _run(issue, graph, reset)
    from test_gpu_layernorm import ln_check
    for k in range(1, STEPS + 1):
        ln_check(X[k], H[k], X[k - 1], H[k - 1], w, b, wl.eps, "bf16", f"layernorm step {k}")


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_qk_chain_in_place(graph):
    """Fused Q+K head norm chained in place on a packed projection (snapshot
    scheme as above; value heads untouched throughout)."""
    wl = W.QK_WORKLOADS["qk_bf16_8192tok_q32_k8_v8_hd128"]
    tokens = 2048
    qkv0, q_w, k_w = W.make_qk_inputs(wl, seed=5, device=DEV, tokens=tokens)
    A = qkv0.clone()
    B = [qkv0.clone() for _ in range(STEPS)]
    span = (wl.q_heads + wl.k_heads) * wl.head_dim

    def issue():
        for k in range(STEPS):
            R.qk_norm(A, wl.q_heads, wl.k_heads, wl.head_dim, q_w=q_w, k_w=k_w, eps=wl.eps, out=B[k])
            R.qk_norm(A, wl.q_heads, wl.k_heads, wl.head_dim, q_w=q_w, k_w=k_w, eps=wl.eps, out=A)

    def reset():
        A.copy_(qkv0)
        for t in B:
            t.copy_(qkv0)

    _run(issue, graph, reset)
    prev = _bits(qkv0)
    qn, kn = _bits(q_w), _bits(k_w)
    for k in range(STEPS):
        qy, ky = oracle.rmsnorm_qk(prev, wl.q_heads, wl.k_heads, wl.head_dim, q_w=qn, k_w=kn, eps=wl.eps,
                                   dtype="bf16", threads=THREADS)
        ref = np.concatenate([qy.reshape(tokens, -1), ky.reshape(tokens, -1)], axis=1)
        got = _bits(B[k])
        ok, rep = parity.compare_y(np.ascontiguousarray(got[:, :span]), ref, "bf16")
        assert ok, f"qk step {k}: {rep}"
        prev = got.copy()
        prev[:, span:] = _bits(qkv0)[:, span:]
    a = _bits(A)
    assert np.array_equal(a[:, :span], prev[:, :span]), "in-place heads differ from their twin"
    assert np.array_equal(a[:, span:], _bits(qkv0)[:, span:]), "value heads were written"
