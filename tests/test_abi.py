"""The C ABI without a GPU: the library loads, exports what the header
declares, plans correctly, and rejects bad arguments before any CUDA call."""
import ctypes
import re

import pytest

import row_reduction_norm_gb300 as R
from row_reduction_norm_gb300 import _native as N
from row_reduction_norm_gb300 import build as B

HEADER = B.os.path.join(B.INCLUDE, "rmsnorm.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:rmsnorm|layernorm)_\w+)\s*\(", text)))


def test_library_builds_and_loads():
    B.build()
    lib = N.load()
    assert "sm_103a" in R.rmsnorm_build_info()
    assert lib is N.load()


def test_every_declared_symbol_is_exported():
    lib = ctypes.CDLL(N.library_path())
    declared = header_functions()
    assert declared == sorted(N.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_plan_struct_layout():
    assert ctypes.sizeof(N.Plan) == 48
    assert N.Plan.grid.offset == 40


def test_strerror_and_limits():
    assert R.rmsnorm_strerror(0) == "ok"
    assert "invalid" in R.rmsnorm_strerror(-1)
    assert R.rmsnorm_max_hidden(N.RMSNORM_BF16) == 65536
    assert R.rmsnorm_max_hidden(N.RMSNORM_F32) == 65536
    assert R.rmsnorm_max_hidden(7) == 0
    assert R.rmsnorm_reg_max_chunks() == 8


def _status(*args):
    return N.rmsnorm_fwd_status(*args)


def test_invalid_arguments_rejected_without_cuda():
    P = 1 << 20   # a fake, aligned address: never dereferenced, checks fail first
    assert _status(None, None, None, P, None, 4, 64, 1e-6, 1, 0) == N.RMSNORM_EINVAL
    assert _status(P, None, None, None, None, 4, 64, 1e-6, 1, 0) == N.RMSNORM_EINVAL
    assert _status(P, None, None, P, None, -1, 64, 1e-6, 1, 0) == N.RMSNORM_EINVAL
    assert _status(P, None, None, P, None, 4, 0, 1e-6, 1, 0) == N.RMSNORM_EINVAL
    assert _status(P, None, None, P, None, 4, 64, 1e-6, 5, 0) == N.RMSNORM_EINVAL
    assert _status(P, None, None, P, None, 4, 64, -1e-6, 1, 0) == N.RMSNORM_EINVAL
    assert _status(P, None, None, P, None, 4, 64, float("inf"), 1, 0) == N.RMSNORM_EINVAL
    assert _status(P, P, None, P, None, 4, 64, 1e-6, 1, 0) == N.RMSNORM_EINVAL
    assert _status(P, None, None, P, P, 4, 64, 1e-6, 1, 0) == N.RMSNORM_EINVAL
    assert _status(P, None, None, P, None, 4, 65537, 1e-6, 1, 0) == N.RMSNORM_EUNSUPPORTED
    assert _status(P + 1, None, None, P, None, 4, 64, 1e-6, 1, 0) == N.RMSNORM_EINVAL   # odd address
    assert _status(P, None, P + 2, P, None, 4, 64, 1e-6, 0, 0) == N.RMSNORM_EINVAL     # f32 needs 4
    assert _status(P, None, None, P, None, 1 << 62, 64, 1e-6, 1, 0) == N.RMSNORM_EINVAL  # overflow
    # rows == 0 is a successful no-op (no CUDA call, no pointer read: NULL is fine)
    assert _status(P, None, None, P, None, 0, 64, 1e-6, 1, 0) == N.RMSNORM_OK
    assert _status(None, None, None, None, None, 0, 64, 1e-6, 1, 0) == N.RMSNORM_OK
    assert _status(None, None, None, None, None, 0, 64, -1.0, 1, 0) == N.RMSNORM_EINVAL


HIDDENS = [1, 2, 7, 8, 16, 31, 33, 64, 127, 128, 256, 576, 1000, 1024, 1025, 2048, 3072, 4096,
           5120, 7168, 8192, 12288, 16384, 32768, 65536]


@pytest.mark.parametrize("dtype", [N.RMSNORM_BF16, N.RMSNORM_F32])
@pytest.mark.parametrize("hidden", HIDDENS)
def test_plan_properties(dtype, hidden):
    V = 8 if dtype == N.RMSNORM_BF16 else 4
    esz = 2 if dtype == N.RMSNORM_BF16 else 4
    for vec_ok in (True, False):
        if vec_ok and (hidden * esz) % 16:
            with pytest.raises(N.RmsNormError):
                R.rmsnorm_plan(10, hidden, dtype, True, 152, 2)
            continue
        plans = [R.rmsnorm_plan(rows, hidden, dtype, vec_ok, 152, 2) for rows in (1, 7, 1000, 10 ** 6)]
        huge = R.rmsnorm_plan(10 ** 12, hidden, dtype, vec_ok, 152, 2)
        tma = huge.kernel == N.RMSNORM_KERNEL_TMA
        assert huge.persistent == 1 and huge.grid == (152 * 2 if tma else 152 * 2 * 4096)
        if huge.kernel == N.RMSNORM_KERNEL_REG:
            assert huge.regime == N.RMSNORM_REGIME_PERSISTENT
        sched = {(p.kernel, p.threads_per_row, p.vec_elems, p.block_threads) for p in plans}
        assert len(sched) == 1, "the per-row schedule must not depend on the row count"
        if plans[0].kernel == N.RMSNORM_KERNEL_REG:
            # only the chunk count may follow the row count: a power of two for
            # a single wave of blocks of rows wider than a warp, the exact fit
            # (3 or 6) beyond, and for rows of a warp or less in every launch
            gt = plans[0].threads_per_row
            need = -(-(hidden // V) // gt)
            pow2 = 1
            while pow2 < need:
                pow2 *= 2
            exact = 3 if need == 3 else 6 if need in (5, 6) else pow2
            for rows, p in zip((1, 7, 1000, 10 ** 6), plans):
                waves = -(-rows // (p.block_threads // gt)) > 152 * 2
                assert p.chunks_per_thread == (exact if waves or gt <= 32 else pow2), (rows, p)
        cap = 152 * 2 if tma else 152 * 2 * 4096
        for rows, p in zip((1, 7, 1000, 10 ** 6), plans):
            row_blocks = -(-rows // p.rows_per_block)
            assert 1 <= p.grid <= min(row_blocks, cap)
            assert p.persistent == (row_blocks > cap)
            assert p.pdl == 1
            if p.kernel == N.RMSNORM_KERNEL_REG:
                assert vec_ok and p.vec_elems == V
                gt, ch = p.threads_per_row, p.chunks_per_thread
                assert gt * ch * V >= hidden and gt & (gt - 1) == 0 and 4 <= gt <= 512
                assert ch in (1, 2, 3, 4, 6, 8)
                assert p.block_threads == max(gt, 256)
                # decode batches: one warp of rows a block while that needs no more blocks than SMs
                want = 1 if gt >= 32 else 32 // gt
                spread = -(-rows // want) <= 152 and want < p.block_threads // gt
                assert p.rows_per_block == (want if spread else p.block_threads // gt), (rows, p)
                want = (N.RMSNORM_REGIME_PERSISTENT if p.persistent else
                        N.RMSNORM_REGIME_WARP if gt <= 32 else N.RMSNORM_REGIME_CTA)
                assert p.regime == want
            elif p.kernel == N.RMSNORM_KERNEL_TMA:
                # rows past 256 threads x 8 chunks that fit the rings
                assert vec_ok and p.vec_elems == V and hidden * esz > 256 * 8 * 16
                assert p.chunks_per_thread == (2 if dtype == N.RMSNORM_F32 and hidden * esz <= 80 * 1024 else 4)
                assert N.tma_rings(hidden * esz, p.chunks_per_thread, False, True) is not None
                assert p.regime == N.RMSNORM_REGIME_SMEM
                assert (p.threads_per_row, p.block_threads, p.rows_per_block) == (512, 608, 1)
                assert N.tma_rings(hidden * esz, p.chunks_per_thread, True, True) is not None
            else:
                assert p.kernel == N.RMSNORM_KERNEL_LOOP and p.regime == N.RMSNORM_REGIME_LOOPED
                assert p.vec_elems == (V if vec_ok else 1)
                units = hidden // p.vec_elems
                assert -(-units // p.block_threads) * p.vec_elems <= 64
        if not vec_ok:
            assert plans[0].kernel == N.RMSNORM_KERNEL_LOOP


@pytest.mark.parametrize("dtype,hidden,kernel", [
    (N.RMSNORM_BF16, 16384, N.RMSNORM_KERNEL_REG), (N.RMSNORM_BF16, 16392, N.RMSNORM_KERNEL_TMA),
    (N.RMSNORM_BF16, 40960, N.RMSNORM_KERNEL_TMA), (N.RMSNORM_BF16, 40968, N.RMSNORM_KERNEL_TMA),
    (N.RMSNORM_BF16, 65536, N.RMSNORM_KERNEL_TMA),
    (N.RMSNORM_F32, 8192, N.RMSNORM_KERNEL_REG), (N.RMSNORM_F32, 8196, N.RMSNORM_KERNEL_TMA),
    (N.RMSNORM_F32, 20480, N.RMSNORM_KERNEL_TMA), (N.RMSNORM_F32, 20484, N.RMSNORM_KERNEL_TMA),
    (N.RMSNORM_F32, 49152, N.RMSNORM_KERNEL_TMA), (N.RMSNORM_F32, 49156, N.RMSNORM_KERNEL_LOOP),
    (N.RMSNORM_F32, 65536, N.RMSNORM_KERNEL_LOOP)])
def test_long_rows_go_to_the_shared_memory_ring(dtype, hidden, kernel):
    """Rows past 256 threads x 8 chunks of 16 bytes (32 KB) take the
    bulk-copy kernel: with 16 KB pieces while the weight stays resident beside
    the row (80 KB), past that (planned without a residual, as this call
    does) with 32 KB pieces while the row fits (192 KB); the two-pass kernel
    beyond that or when unaligned; rows of 16 to 32 KB take 256 threads x 8
    chunks."""
    p = R.rmsnorm_plan(1000, hidden, dtype, True, 152, 1)
    assert p.kernel == kernel
    if kernel == N.RMSNORM_KERNEL_REG:
        assert (p.threads_per_row, p.chunks_per_thread) == (256, 8)
    if kernel == N.RMSNORM_KERNEL_TMA:
        esz = 2 if dtype == N.RMSNORM_BF16 else 4
        # planned without a residual: 32 KB pieces for bf16 and past 80 KB
        assert p.chunks_per_thread == (2 if dtype == N.RMSNORM_F32 and hidden * esz <= 80 * 1024 else 4)
        assert p.grid == 152 and p.persistent == 1
        assert R.rmsnorm_plan(100, hidden, dtype, True, 152, 1).grid == 100
    assert R.rmsnorm_plan(1000, hidden, dtype, False, 152, 1).kernel == N.RMSNORM_KERNEL_LOOP


def test_tma_plan_validation_without_cuda():
    P = 1 << 20
    good = R.rmsnorm_plan(4, 40000, N.RMSNORM_BF16, True, 152, 1)
    assert good.kernel == N.RMSNORM_KERNEL_TMA

    def st(plan, hidden=40000, dtype=N.RMSNORM_BF16, res=None, x=P):
        return N.rmsnorm_fwd_plan_status(x, res, None, P, res, 4, hidden, 1e-6, dtype, plan, 0)

    for field, value in (("chunks_per_thread", 3), ("chunks_per_thread", 8), ("threads_per_row", 256),
                         ("block_threads", 544), ("rows_per_block", 2), ("vec_elems", 1)):
        q = good.copy()
        setattr(q, field, value)
        assert st(q) == N.RMSNORM_EINVAL, field
    # 65536 fp32 (256 KB) does not fit the x ring; 57344 fp32 (224 KB) fits it
    # only without a residual (a weight then takes no slot: it is read from
    # global memory)
    q = good.copy()
    q.vec_elems = 4
    assert st(q, hidden=65536, dtype=N.RMSNORM_F32) == N.RMSNORM_EINVAL
    for res, w, status in ((None, None, N.RMSNORM_OK), (None, P, N.RMSNORM_OK), (P, None, N.RMSNORM_EINVAL),
                           (P, P, N.RMSNORM_EINVAL)):   # rows = 0: validation only
        assert N.rmsnorm_fwd_plan_status(P, res, w, P, res, 0, 57344, 1e-6, N.RMSNORM_F32, q, 0) == status
    assert N.tma_rings(57344 * 4, 4, False, True) == (7, 0, 0)        # no weight ring
    assert N.tma_rings(65536 * 2, 4, False, True) == (7, 0, 0)
    assert N.tma_rings(32768 * 2, 4, False, True) == (5, 0, 2)        # resident: two spare x slots
    assert N.tma_rings(40960 * 2, 2, True, True) == (7, 2, 5)
    # 32 KB pieces: 7 slots, 40000 bf16 (80 KB) fits, a misaligned x does not
    q = good.copy()
    q.chunks_per_thread = 4
    assert st(q, x=P + 2) == N.RMSNORM_EINVAL
    # rows == 0 validates the plan and launches nothing
    assert N.rmsnorm_fwd_plan_status(P, None, None, P, None, 0, 40000, 1e-6, 1, good, 0) == N.RMSNORM_OK
    # block-scaled outputs run on it with 16 KB pieces only (rows = 0: validation only)
    q = good.copy()
    q.chunks_per_thread = 2
    assert N.rmsnorm_fwd_mxfp8_status(P, None, None, P, P, None, 0, 40000, 1e-6, 0.0, 1, q) == N.RMSNORM_OK
    assert N.rmsnorm_fwd_nvfp4_status(P, None, None, P, P, None, 0, 40000, 1e-6, 0.0, 1.0, 1, q) == N.RMSNORM_OK
    q.chunks_per_thread = 4
    assert N.rmsnorm_fwd_mxfp8_status(P, None, None, P, P, None, 0, 40000, 1e-6, 0.0, 1, q) == N.RMSNORM_EINVAL
    assert N.rmsnorm_fwd_nvfp4_status(P, None, None, P, P, None, 0, 40000, 1e-6, 0.0, 1.0, 1, q) == N.RMSNORM_EINVAL
    # LayerNorm and head rows have no bulk-copy kernel
    assert N.layernorm_fwd_status(P, None, None, None, P, None, 4, 40000, 1e-5, 1, good) == N.RMSNORM_EINVAL
    assert N.rmsnorm_qk_fwd_status(P, P, 4, 40000, 40000, 1, 0, 40000, None, None, 0.0, 1e-6, 1,
                                   good) == N.RMSNORM_EINVAL


@pytest.mark.parametrize("pc", [1, 2, 4])
@pytest.mark.parametrize("res", [False, True])
@pytest.mark.parametrize("w", [False, True])
def test_tma_ring_rule_matches_the_library(pc, res, w):
    """The Python restatement of the ring sizing accepts exactly the plans the
    library accepts (rows = 0 validates a plan and launches nothing)."""
    P = 1 << 20
    plan = R.rmsnorm_plan(4, 40000, N.RMSNORM_BF16, True, 152, 1)
    plan.chunks_per_thread = pc
    for dtype, esz in ((N.RMSNORM_BF16, 2), (N.RMSNORM_F32, 4)):
        plan.vec_elems = 16 // esz
        for hidden in range(4096, 65537, 4096 - 8):
            hidden -= hidden % 8
            want = N.tma_rings(hidden * esz, pc, res, w) is not None
            got = N.rmsnorm_fwd_plan_status(P, P if res else None, P if w else None, P, P if res else None, 0,
                                            hidden, 1e-6, dtype, plan, 0) == N.RMSNORM_OK
            assert got == want, (dtype, hidden)


def _cluster_expected(hidden, dtype):
    """(chunks_per_thread, cluster_ctas) of the cluster rule: 256-thread
    blocks of 16 KB slices, as few as cover the row; four 20 KB slices where
    that takes five (rows of 64 to 80 KB); 32 KB slices for fp32 rows the
    eight-block cap of 16 KB slices cannot cover."""
    V = 8 if dtype == N.RMSNORM_BF16 else 4
    units = hidden // V
    ch = 4 if units <= 8 * 256 * 4 else 8
    if ch == 4 and -(-units // 1024) == 5:
        ch = 5
    return ch, -(-units // (256 * ch))


@pytest.mark.parametrize("dtype", [N.RMSNORM_BF16, N.RMSNORM_F32])
def test_residual_rows_past_32kb_take_the_cluster_kernel(dtype):
    """With a residual, aligned rows past 32 KB run on the cluster kernel,
    one cluster a row; shorter rows, unaligned rows and rows without a
    residual keep rmsnorm_plan's plan."""
    esz = 2 if dtype == N.RMSNORM_BF16 else 4
    V = 16 // esz
    edge = [32768 // esz, 32768 // esz + V, 131072 // esz, 131072 // esz + V, 65536]
    hiddens = sorted(set(list(range(V, 65537, 1000 - 1000 % V)) + [h for h in edge if h <= 65536]))
    for hidden in hiddens:
        for rows in (0, 1, 1000, 10 ** 6):
            p = R.rmsnorm_plan_ex(rows, hidden, dtype, True, True, 152, 4)
            q = R.rmsnorm_plan(rows, hidden, dtype, True, 152, 4)
            assert R.rmsnorm_plan_ex(rows, hidden, dtype, True, False, 152, 4).as_dict() == q.as_dict()
            assert R.rmsnorm_plan_ex(rows, hidden, dtype, False, True, 152, 4).as_dict() == \
                R.rmsnorm_plan(rows, hidden, dtype, False, 152, 4).as_dict()
            if hidden * esz <= 32768:
                assert p.as_dict() == q.as_dict(), hidden
                assert q.cluster_ctas == 0
                continue
            ch, ctas = _cluster_expected(hidden, dtype)
            assert 2 <= ctas <= 8 and (ctas - 1) * 256 * ch * V < hidden <= ctas * 256 * ch * V
            assert dtype == N.RMSNORM_F32 or ch in (4, 5)
            assert ch != 5 or (ctas == 4 and 64 * 1024 < hidden * esz <= 80 * 1024)
            assert (p.kernel, p.regime) == (N.RMSNORM_KERNEL_CLUSTER, N.RMSNORM_REGIME_CLUSTER)
            assert (p.chunks_per_thread, p.cluster_ctas, p.threads_per_row) == (ch, ctas, 256 * ctas)
            assert (p.vec_elems, p.block_threads, p.rows_per_block) == (V, 256, 1)
            assert (p.grid, p.persistent, p.pdl) == (rows * ctas, 0, 1)
            assert q.kernel in (N.RMSNORM_KERNEL_TMA, N.RMSNORM_KERNEL_LOOP) and q.cluster_ctas == 0
    with pytest.raises(N.RmsNormError):
        R.rmsnorm_plan_ex(4, 40960, dtype, True, 2, 152, 4)


def test_cluster_plan_validation_without_cuda():
    """A forced cluster plan is checked before any CUDA call (rows = 0
    validates and launches nothing; a bad plan is refused whatever rows is)."""
    P = 1 << 20
    OK, EINVAL = N.RMSNORM_OK, N.RMSNORM_EINVAL
    good = R.rmsnorm_plan_ex(4, 40960, N.RMSNORM_BF16, True, True, 152, 4)
    assert (good.kernel, good.cluster_ctas, good.chunks_per_thread, good.grid) == (N.RMSNORM_KERNEL_CLUSTER, 4, 5, 16)

    def st(plan, hidden=40960, dtype=N.RMSNORM_BF16, res=P, rows=0, w=None):
        return N.rmsnorm_fwd_plan_status(P, res, w, P, res, rows, hidden, 1e-6, dtype, plan, 0)

    assert st(good) == OK and st(good, w=P) == OK
    # more blocks than the row needs: the extra slices are past the row end
    for c in (5, 6, 7, 8):
        q = good.copy()
        q.cluster_ctas, q.threads_per_row, q.grid = c, 256 * c, 4 * c
        assert st(q) == OK, c
    bad = []
    for field, value in (("chunks_per_thread", 8), ("chunks_per_thread", 2), ("block_threads", 512),
                         ("rows_per_block", 2), ("vec_elems", 4), ("threads_per_row", 256 * 6),
                         ("cluster_ctas", 0), ("cluster_ctas", 1), ("cluster_ctas", 9), ("chunks_per_thread", 3)):
        q = good.copy()
        setattr(q, field, value)
        bad.append(q)
    q = good.copy()
    q.chunks_per_thread = 4                              # 4 x 16 KB slices do not cover 80 KB
    bad.append(q)
    q = good.copy()
    q.cluster_ctas, q.threads_per_row = 3, 768           # nor do 3 x 20 KB
    bad.append(q)
    for q in bad:
        assert st(q) == EINVAL, q.as_dict()
    assert st(good, res=None) == EINVAL                  # compiled for rows with a residual
    q = good.copy()
    q.grid = 21                                          # not a whole number of clusters
    assert st(q, rows=4) == EINVAL
    # fp32: 32 KB slices, 8 blocks for 65536 elements; 16 KB slices do not cover them
    f = R.rmsnorm_plan_ex(4, 65536, N.RMSNORM_F32, True, True, 152, 4)
    assert (f.chunks_per_thread, f.cluster_ctas) == (8, 8)
    assert st(f, hidden=65536, dtype=N.RMSNORM_F32) == OK
    q = f.copy()
    q.chunks_per_thread = 4
    assert st(q, hidden=65536, dtype=N.RMSNORM_F32) == EINVAL
    assert st(q, hidden=32768, dtype=N.RMSNORM_F32) == OK
    # weight forms: bias and the cast order (bf16) run on it
    assert N.rmsnorm_fwd_ex_status(P, P, P, P, P, 0, 40960, 1e-6, 1.0, N.RMSNORM_BF16, good) == OK
    assert N.rmsnorm_fwd_cast_status(P, P, P, P, P, 0, 40960, 1e-6, N.RMSNORM_BF16, good) == OK
    # no block-scaled, LayerNorm or head-row form of it
    assert N.rmsnorm_fwd_mxfp8_status(P, P, None, P, P, P, 0, 40960, 1e-6, 0.0, 1, good) == EINVAL
    assert N.rmsnorm_fwd_nvfp4_status(P, P, None, P, P, P, 0, 40960, 1e-6, 0.0, 1.0, 1, good) == EINVAL
    assert N.layernorm_fwd_status(P, P, None, None, P, P, 0, 40960, 1e-5, 1, good) == EINVAL
    assert N.rmsnorm_qk_fwd_status(P, P, 4, 40960, 40960, 1, 0, 40960, None, None, 0.0, 1e-6, 1,
                                   good) == EINVAL
    # cluster_ctas belongs to cluster plans only
    reg = R.rmsnorm_plan(4, 576, N.RMSNORM_BF16, True, 152, 4)
    reg.cluster_ctas = 2
    assert st(reg, hidden=576, res=None) == EINVAL


def test_host_call_workspace_and_validation_without_cuda():
    """rmsnorm_fwd_host's workspace size (the weight, then two halves of
    chunk_rows rows of x and y, and of residual and residual_out with one,
    every part on a 256-byte boundary) and its argument checks, which all
    return before any CUDA call."""
    up = lambda v: -(-v // 256) * 256
    for dtype, esz in ((N.RMSNORM_BF16, 2), (N.RMSNORM_F32, 4)):
        for chunk, hidden, res in ((1, 1, False), (7, 576, True), (4096, 8192, True), (3, 65536, False)):
            rb = hidden * esz
            want = up(rb) + 2 * (4 if res else 2) * up(chunk * rb)
            assert R.rmsnorm_host_workspace_bytes(chunk, hidden, dtype, res) == want
    W = N.load().rmsnorm_host_workspace_bytes
    assert W(0, 64, 1, 0) == N.RMSNORM_EINVAL and W(4, 0, 1, 0) == N.RMSNORM_EINVAL
    assert W(4, 64, 7, 0) == N.RMSNORM_EINVAL and W(4, 64, 1, 2) == N.RMSNORM_EINVAL
    assert W(4, 65537, 1, 0) == N.RMSNORM_EUNSUPPORTED
    assert W(1 << 60, 65536, 0, 1) == N.RMSNORM_EINVAL      # overflows

    P, H = 1 << 20, 1 << 21                                  # stand-in addresses (never touched)
    need = R.rmsnorm_host_workspace_bytes(16, 1024, N.RMSNORM_BF16, True)

    def st(x=H, r=H, w=H, y=H, h=H, rows=100, hidden=1024, eps=1e-6, dtype=N.RMSNORM_BF16, ws=P, nbytes=need,
           chunk=16):
        return N.rmsnorm_fwd_host_status(x, r, w, y, h, rows, hidden, eps, dtype, ws, nbytes, chunk, 0)

    assert st(rows=0, x=None, r=None, w=None, y=None, h=None, ws=None, nbytes=0) == N.RMSNORM_OK
    EINVAL = N.RMSNORM_EINVAL
    assert st(chunk=0) == EINVAL
    assert st(ws=None) == EINVAL and st(ws=P + 16) == EINVAL and st(nbytes=need - 1) == EINVAL
    assert st(x=None) == EINVAL and st(y=None) == EINVAL
    assert st(h=None) == EINVAL and st(r=None) == EINVAL     # residual and residual_out go together
    assert st(eps=-1.0) == EINVAL and st(dtype=5) == EINVAL and st(rows=-1) == EINVAL
    assert st(hidden=65537) == N.RMSNORM_EUNSUPPORTED
    # without a residual the smaller workspace is enough
    small = R.rmsnorm_host_workspace_bytes(16, 1024, N.RMSNORM_BF16, False)
    assert small < need
    assert st(r=None, h=None, nbytes=small - 1) == EINVAL


def _sum_depth(plan, hidden, dtype):
    """Rounding steps a square passes through on its way into the row's sum,
    for the planned kernel (the count the fp32 tolerance in parity.py is
    derived from): sequential per-accumulator steps, then the fixed trees."""
    V = 8 if dtype == N.RMSNORM_BF16 else 4
    lg = lambda n: max(0, (n - 1).bit_length())
    k, gt, ch = plan.kernel, plan.threads_per_row, plan.chunks_per_thread
    if k == N.RMSNORM_KERNEL_REG:
        return ch + lg(V) + lg(min(gt, 32)) + lg(max(1, gt // 32))
    if k == N.RMSNORM_KERNEL_CLUSTER:
        return ch + lg(V) + 5 + lg(256 // 32) + lg(8)
    if k == N.RMSNORM_KERNEL_TMA:
        return -(-(hidden // V) // 512) + lg(V) + 5 + lg(512 // 32)
    assert k == N.RMSNORM_KERNEL_LOOP
    ve = plan.vec_elems
    units = hidden // ve
    terms = -(-units // plan.block_threads) * ve       # a thread's elements
    return -(-terms // 8) + 3 + 5 + lg(plan.block_threads // 32)


@pytest.mark.parametrize("dtype", [N.RMSNORM_BF16, N.RMSNORM_F32])
def test_planned_sum_trees_stay_within_the_tolerance_derivation(dtype):
    """Every plan the planner makes keeps the fp32 sum of squares within the
    depth the tolerance is derived from: 21 levels for the register, cluster
    and two-pass kernels, 35 for the bulk-copy kernel (see tests/parity.py)."""
    esz = 2 if dtype == N.RMSNORM_BF16 else 4
    worst = {}
    edges = [16 // esz * k for k in (1, 512, 2048, 2049, 8192, 16384)]
    for hidden in list(range(1, 65537, 61)) + [h for h in edges if h <= 65536]:
        for vec_ok in (True, False):
            if vec_ok and (hidden * esz) % 16:
                continue
            for res in (False, True):
                for rows in (1, 4096):
                    p = R.rmsnorm_plan_ex(rows, hidden, dtype, vec_ok, res, 152, 4)
                    d = _sum_depth(p, hidden, dtype)
                    limit = 35 if p.kernel == N.RMSNORM_KERNEL_TMA else 21
                    assert d <= limit, (hidden, vec_ok, res, rows, p.as_dict(), d)
                    worst[p.kernel] = max(worst.get(p.kernel, 0), d)
    assert set(worst) == {N.RMSNORM_KERNEL_REG, N.RMSNORM_KERNEL_CLUSTER, N.RMSNORM_KERNEL_TMA,
                          N.RMSNORM_KERNEL_LOOP}


def test_layernorm_register_blocks_are_four_warps_or_the_row():
    """LayerNorm register plans use blocks of max(threads_per_row, 128)
    threads; a plan with the RMSNorm block size is refused (rows = 0:
    validation only, no CUDA call)."""
    P = 1 << 20
    p = R.rmsnorm_plan(4, 768, N.RMSNORM_BF16, True, 152, 1)
    p.threads_per_row, p.chunks_per_thread, p.block_threads, p.rows_per_block = 32, 3, 128, 4
    assert N.layernorm_fwd_status(P, None, P, P, P, None, 0, 768, 1e-5, 1, p) == N.RMSNORM_OK
    q = p.copy()
    q.block_threads, q.rows_per_block = 256, 8
    assert N.layernorm_fwd_status(P, None, P, P, P, None, 0, 768, 1e-5, 1, q) == N.RMSNORM_EINVAL
    # RMSNorm keeps 256-thread blocks
    assert N.rmsnorm_fwd_plan_status(P, None, P, P, None, 0, 768, 1e-5, 1, q, 0) == N.RMSNORM_OK
    assert N.rmsnorm_fwd_plan_status(P, None, P, P, None, 0, 768, 1e-5, 1, p, 0) == N.RMSNORM_EINVAL
    big = p.copy()
    big.threads_per_row, big.chunks_per_thread, big.block_threads, big.rows_per_block = 128, 4, 128, 1
    assert N.layernorm_fwd_status(P, None, P, P, P, None, 0, 4096, 1e-5, 1, big) == N.RMSNORM_OK


def test_qk_norm_is_warp_regime_and_large_rows_cta():
    qk = R.rmsnorm_plan(1024, 128, N.RMSNORM_BF16, True, 152, 4)
    assert qk.regime == N.RMSNORM_REGIME_WARP and qk.threads_per_row <= 32
    big = R.rmsnorm_plan(100, 8192, N.RMSNORM_BF16, True, 152, 4)
    assert big.regime == N.RMSNORM_REGIME_CTA and big.threads_per_row > 32


def test_regime_query_rejects_bad_input_without_cuda():
    # argument checks come before any CUDA call; a valid query needs a device
    assert N.rmsnorm_regime_status(-1, 576, N.RMSNORM_BF16) == N.RMSNORM_EINVAL
    assert N.rmsnorm_regime_status(4, 0, N.RMSNORM_BF16) == N.RMSNORM_EINVAL
    assert N.rmsnorm_regime_status(4, 576, 7) == N.RMSNORM_EINVAL
    assert N.rmsnorm_regime_status(4, 65537, N.RMSNORM_BF16) == N.RMSNORM_EUNSUPPORTED
    assert N.rmsnorm_regime_status(1 << 62, 576, N.RMSNORM_BF16) == N.RMSNORM_EINVAL
    st = N.rmsnorm_regime_status(4096, 576, N.RMSNORM_BF16)
    assert st in (N.RMSNORM_REGIME_WARP, N.RMSNORM_ECUDA)


def test_rows_per_block_validation_without_cuda():
    """A register plan may hold 1 .. block_threads / threads_per_row rows a
    block (RMSNorm); 0 or more than its row slots is refused (rows = 0:
    validation only)."""
    P = 1 << 20
    p = R.rmsnorm_plan(4096, 576, N.RMSNORM_BF16, True, 152, 4)
    assert p.kernel == N.RMSNORM_KERNEL_REG and p.rows_per_block == 8
    for rpb, want in ((1, N.RMSNORM_OK), (5, N.RMSNORM_OK), (8, N.RMSNORM_OK), (0, N.RMSNORM_EINVAL),
                      (9, N.RMSNORM_EINVAL), (-1, N.RMSNORM_EINVAL)):
        q = p.copy()
        q.rows_per_block = rpb
        assert N.rmsnorm_fwd_plan_status(P, None, P, P, None, 0, 576, 1e-6, 1, q, 0) == want, rpb
        h = q.copy()
        h.chunks_per_thread = 4   # head rows have no odd chunk counts
        assert N.rmsnorm_qk_fwd_status(P, P, 0, 576, 576, 1, 0, 576, None, None, 0.0, 1e-6, 1, h) == want, rpb


def test_plan_rejects_bad_input():
    with pytest.raises(N.RmsNormError):
        R.rmsnorm_plan(-1, 128, 1, True, 152, 1)
    with pytest.raises(N.RmsNormError) as e:
        R.rmsnorm_plan(1, 1 << 20, 1, True, 152, 1)
    assert e.value.status == N.RMSNORM_EUNSUPPORTED


def test_fwd_plan_validation_without_cuda():
    P = 1 << 20
    p = R.rmsnorm_plan(4, 64, N.RMSNORM_BF16, True, 152, 1)
    q = p.copy()
    q.threads_per_row = 3
    assert N.rmsnorm_fwd_plan_status(P, None, None, P, None, 4, 64, 1e-6, 1, q, 0) == N.RMSNORM_EINVAL
    q = p.copy()
    q.chunks_per_thread = 16
    assert N.rmsnorm_fwd_plan_status(P, None, None, P, None, 4, 64, 1e-6, 1, q, 0) == N.RMSNORM_EINVAL
    q = p.copy()
    q.grid = 0
    assert N.rmsnorm_fwd_plan_status(P, None, None, P, None, 4, 64, 1e-6, 1, q, 0) == N.RMSNORM_EINVAL
    # a vector plan on a misaligned pointer
    assert N.rmsnorm_fwd_plan_status(P + 2, None, None, P, None, 4, 64, 1e-6, 1, p, 0) == N.RMSNORM_EINVAL
    assert N.rmsnorm_fwd_plan_status(P, None, None, P, None, 4, 64, 1e-6, 1, None, 0) == N.RMSNORM_EINVAL
    # rows == 0 with a valid plan: no-op
    assert N.rmsnorm_fwd_plan_status(P, None, None, P, None, 0, 64, 1e-6, 1, p, 0) == N.RMSNORM_OK


def test_torch_api_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        R.rms_norm(x)


def _qk(*a):
    return N.rmsnorm_qk_fwd_status(*a)


def test_qk_and_ex_arguments_rejected_without_cuda():
    P = 1 << 20
    # x, y, tokens, xs, ys, qh, kh, hd, q_w, k_w, bias, eps, dtype
    ok = (P, P, 4, 48 * 128, 48 * 128, 32, 8, 128, P, P, 0.0, 1e-6, 1)
    bad = [
        (P, P, 4, 48 * 128, 48 * 128, -1, 8, 128, P, P, 0.0, 1e-6, 1),          # negative heads
        (P, P, 4, 48 * 128, 48 * 128, 0, 0, 128, P, P, 0.0, 1e-6, 1),          # no heads
        (P, P, 4, 39 * 128, 48 * 128, 32, 8, 128, P, P, 0.0, 1e-6, 1),         # x stride too short
        (P, P, 4, 48 * 128, 39 * 128, 32, 8, 128, P, P, 0.0, 1e-6, 1),         # y stride too short
        (P, P, 4, 48 * 128, 64 * 128, 32, 8, 128, P, P, 0.0, 1e-6, 1),         # in place, strides differ
        (P, P, 4, 48 * 128, 48 * 128, 32, 8, 128, P, None, 0.0, 1e-6, 1),      # one weight only
        (P, P, 4, 48 * 128, 48 * 128, 32, 8, 128, None, None, 1.0, 1e-6, 1),   # bias without weights
        (P, P, 4, 48 * 128, 48 * 128, 32, 8, 0, P, P, 0.0, 1e-6, 1),           # head_dim 0
        (P, P, 4, 48 * 128, 48 * 128, 32, 8, 128, P, P, float("nan"), 1e-6, 1),  # bias not finite
        (P, P, -1, 48 * 128, 48 * 128, 32, 8, 128, P, P, 0.0, 1e-6, 1),        # negative tokens
        (None, P, 4, 48 * 128, 48 * 128, 32, 8, 128, P, P, 0.0, 1e-6, 1),      # null x
        (P + 1, P, 4, 48 * 128, 48 * 128, 32, 8, 128, P, P, 0.0, 1e-6, 1),     # misaligned element
    ]
    for a in bad:
        assert _qk(*a) == N.RMSNORM_EINVAL, a
    assert _qk(P, P, 4, 48 * 128, 48 * 128, 32, 8, 1 << 17, P, P, 0.0, 1e-6, 1) == N.RMSNORM_EUNSUPPORTED
    # zero tokens: a successful no-op, pointers unused
    assert _qk(None, None, 0, 48 * 128, 48 * 128, 32, 8, 128, None, None, 0.0, 1e-6, 1) == N.RMSNORM_OK
    # weight bias needs a weight; non-finite bias rejected
    assert N.rmsnorm_fwd_ex_status(P, None, None, P, None, 4, 64, 1e-6, 1.0, 1) == N.RMSNORM_EINVAL
    assert N.rmsnorm_fwd_ex_status(P, None, P, P, None, 4, 64, 1e-6, float("inf"), 1) == N.RMSNORM_EINVAL
    assert N.rmsnorm_fwd_ex_status(P, None, P, P, None, 0, 64, 1e-6, 1.0, 1) == N.RMSNORM_OK
    bad_plan = R.rmsnorm_plan(4, 64, 1, True, 152, 1)
    bad_plan.threads_per_row = 64    # head rows allow at most 32 threads per row
    bad_plan.block_threads = 256
    bad_plan.rows_per_block = 4
    bad_plan.chunks_per_thread = 1
    assert N.rmsnorm_qk_fwd_status(P, P, 4, 48 * 512, 48 * 512, 32, 8, 512, P, P, 0.0, 1e-6, 1,
                                   bad_plan) == N.RMSNORM_EINVAL
    del ok


def test_cast_arguments_rejected_without_cuda():
    P = 1 << 20
    f = N.rmsnorm_fwd_cast_status
    # x, residual, w, y, residual_out, rows, hidden, eps, dtype
    bad = [
        (P, None, P, P, None, 4, 64, -1.0, 1),            # negative eps
        (P, None, P, P, None, 4, 64, float("nan"), 1),    # eps not finite
        (P, None, P, P, None, 4, 64, 1e-6, 2),            # unknown dtype
        (P, P, P, P, None, 4, 64, 1e-6, 1),               # residual without residual_out
        (None, None, P, P, None, 4, 64, 1e-6, 1),         # null x
        (P, None, P, P, None, 4, 0, 1e-6, 1),             # hidden 0
        (P, None, P, P, None, -1, 64, 1e-6, 1),           # negative rows
        (P + 1, None, P, P, None, 4, 64, 1e-6, 1),        # misaligned element
    ]
    for a in bad:
        assert f(*a) == N.RMSNORM_EINVAL, a
    assert f(P, None, P, P, None, 4, 1 << 40, 1e-6, 1) in (N.RMSNORM_EUNSUPPORTED, N.RMSNORM_EINVAL)
    # zero rows: a successful no-op, pointers unused
    assert f(None, None, None, None, None, 0, 64, 1e-6, 1) == N.RMSNORM_OK
    assert f(P, P, P, P, P, 0, 64, 1e-6, 0) == N.RMSNORM_OK


def test_header_is_plain_c_and_links():
    # the boundary as a C caller sees it: the header compiles as strict C99,
    # the program links against the library and calls it (no CUDA work: a
    # zero-row call, a call rejected for its eps, the regime query, which
    # answers the warp regime on a GPU and a CUDA error without one, and the
    # host planner's cluster plan for rows of 80 KB with a residual)
    import os
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not installed")
    from row_reduction_norm_gb300 import build as B
    lib = B.build()
    out_dir = os.path.join(B.BUILD_DIR, "c_abi_check")
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "abi_check.c")
    exe = os.path.join(out_dir, "abi_check")
    with open(src, "w") as f:
        f.write(r'''
#include "rmsnorm.h"
#include <stdio.h>
int main(void) {
    const char *info = rmsnorm_build_info();
    int zero = rmsnorm_fwd(NULL, NULL, NULL, NULL, NULL, 0, 64, 1e-6f, RMSNORM_BF16, NULL);
    int bad = rmsnorm_fwd((const void *)1048576, NULL, NULL, (void *)1048576, NULL, 4, 64, -1.0f,
                          RMSNORM_BF16, NULL);
    int cast = rmsnorm_fwd_cast(NULL, NULL, NULL, NULL, NULL, 0, 64, 1e-6f, RMSNORM_BF16, NULL, NULL);
    int regime_bad = rmsnorm_regime(-1, 576, RMSNORM_BF16);
    int regime = rmsnorm_regime(4096, 576, RMSNORM_BF16);
    rmsnorm_plan_t plan;
    int planned = rmsnorm_plan_ex(100, 40960, RMSNORM_BF16, 1, 1, 152, 4, &plan);
    int cluster = planned == RMSNORM_OK && plan.kernel == RMSNORM_KERNEL_CLUSTER &&
                  plan.regime == RMSNORM_REGIME_CLUSTER && plan.cluster_ctas == 4 &&
                  plan.chunks_per_thread == 5 && plan.grid == 400;
    printf("%d %d %d %d %d %d %d\n", zero, bad, cast, info != NULL, regime_bad,
           regime == RMSNORM_REGIME_WARP || regime == RMSNORM_ECUDA, cluster);
    return 0;
}
''')
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", B.INCLUDE, src,
           "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib), "-Wl,-rpath," + os.path.dirname(lib),
           "-o", exe]
    subprocess.run(cmd, check=True)
    r = subprocess.run([exe], capture_output=True, text=True, check=True)
    assert r.stdout.split() == [str(N.RMSNORM_OK), str(N.RMSNORM_EINVAL), str(N.RMSNORM_OK), "1",
                                str(N.RMSNORM_EINVAL), "1", "1"]
