"""ctypes binding of the C ABI in ``include/rmsnorm.h`` (argument marshalling only).

The functions keep the C names and argument order; pointers are plain
integers (device addresses; host addresses for the tensors of
``rmsnorm_fwd_host``), streams are ``cudaStream_t`` values as integers.
A non-zero status raises ``RmsNormError``.  Nothing here computes any part of
the op: every step runs in the CUDA kernels of ``librmsnorm_gb300.so``, and a
missing library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "librmsnorm_gb300.so")

RMSNORM_F32 = 0
RMSNORM_BF16 = 1

RMSNORM_OK = 0
RMSNORM_EINVAL = -1
RMSNORM_EUNSUPPORTED = -2
RMSNORM_ECUDA = -3

RMSNORM_KERNEL_REG = 0
RMSNORM_KERNEL_LOOP = 1
RMSNORM_KERNEL_TMA = 2
RMSNORM_KERNEL_CLUSTER = 3

RMSNORM_REGIME_WARP = 0
RMSNORM_REGIME_CTA = 1
RMSNORM_REGIME_PERSISTENT = 2
RMSNORM_REGIME_LOOPED = 3
RMSNORM_REGIME_SMEM = 4
RMSNORM_REGIME_CLUSTER = 5

REGIME_NAMES = {0: "warp", 1: "cta", 2: "persistent", 3: "looped", 4: "smem", 5: "cluster"}
KERNEL_NAMES = {0: "reg", 1: "loop", 2: "tma", 3: "cluster"}

# Shape of the bulk-copy (TMA) kernel's block and rings (include/rmsnorm.h).
TMA_THREADS_PER_ROW = 512
TMA_BLOCK_THREADS = 608
TMA_PIECE_CHUNKS = (1, 2, 4)
_TMA_SMEM_BUDGET = 227 * 1024 - 1024
_TMA_BAR_BYTES = 2 * 32 * 8


def tma_rings(row_bytes, pc, res, w):
    """(x, residual, weight) ring slots of the bulk-copy kernel for rows of
    ``row_bytes`` and pieces of ``pc`` chunks a thread, or None when the row
    does not fit -- the rule of ``rmsnorm_plan_t.chunks_per_thread``, restated
    so tests can tell which forced plans are valid.  A weight slot count of 0
    with a weight means the kernel reads the weight from global memory."""
    piece = 512 * 16 * pc
    avail = min(32, (_TMA_SMEM_BUDGET - _TMA_BAR_BYTES) // piece)
    pieces = -(-row_bytes // piece)
    streamed = max(1, avail // 7)
    sr = streamed if res else 0
    sw = pieces if (w and avail - sr - pieces >= pieces + 2) else 0
    sx = avail - sr - sw
    return (sx, sr, sw) if sx >= pieces else None

# Every symbol the header declares (checked by the CPU tests).
EXPORTED = ["rmsnorm_fwd", "rmsnorm_regime", "rmsnorm_plan", "rmsnorm_plan_ex", "rmsnorm_plan_for",
            "rmsnorm_fwd_plan", "rmsnorm_fwd_ex", "rmsnorm_fwd_cast",
            "rmsnorm_qk_fwd", "rmsnorm_qk_plan_for", "rmsnorm_fwd_mxfp8", "rmsnorm_mxfp8_plan_for",
            "rmsnorm_fwd_nvfp4", "rmsnorm_nvfp4_plan_for",
            "layernorm_fwd", "layernorm_plan_for",
            "rmsnorm_fwd_host", "rmsnorm_host_workspace_bytes", "rmsnorm_fwd_host_static",
            "rmsnorm_max_hidden", "rmsnorm_reg_max_chunks", "rmsnorm_wait_timeouts", "rmsnorm_tma_wait_test",
            "rmsnorm_strerror",
            "rmsnorm_build_info"]


class RmsNormError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {rmsnorm_strerror(status)} (status {status})")


class Plan(ctypes.Structure):
    """Mirror of ``rmsnorm_plan_t``."""
    _fields_ = [
        ("kernel", ctypes.c_int32),
        ("regime", ctypes.c_int32),
        ("threads_per_row", ctypes.c_int32),
        ("chunks_per_thread", ctypes.c_int32),
        ("vec_elems", ctypes.c_int32),
        ("block_threads", ctypes.c_int32),
        ("rows_per_block", ctypes.c_int32),
        ("persistent", ctypes.c_int32),
        ("pdl", ctypes.c_int32),
        ("cluster_ctas", ctypes.c_int32),
        ("grid", ctypes.c_int64),
    ]

    def as_dict(self):
        d = {k: getattr(self, k) for k, _ in self._fields_}
        d["kernel_name"] = KERNEL_NAMES.get(self.kernel, "?")
        d["regime_name"] = REGIME_NAMES.get(self.regime, "?")
        return d

    def copy(self):
        p = Plan()
        ctypes.pointer(p)[0] = self
        return p

    def __repr__(self):
        return f"Plan({self.as_dict()})"


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m row_reduction_norm_gb300.build` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        fwd_args = [vp, vp, vp, vp, vp, i64, i64, ctypes.c_float, i32]
        lib.rmsnorm_fwd.argtypes = fwd_args + [vp]
        lib.rmsnorm_fwd.restype = i32
        lib.rmsnorm_fwd_plan.argtypes = fwd_args + [ctypes.POINTER(Plan), vp]
        lib.rmsnorm_fwd_plan.restype = i32
        lib.rmsnorm_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, ctypes.c_float, ctypes.c_float, i32,
                                       ctypes.POINTER(Plan), vp]
        lib.rmsnorm_fwd_ex.restype = i32
        lib.rmsnorm_fwd_cast.argtypes = fwd_args + [ctypes.POINTER(Plan), vp]
        lib.rmsnorm_fwd_cast.restype = i32
        lib.rmsnorm_qk_fwd.argtypes = [vp, vp, i64, i64, i64, ctypes.c_int32, ctypes.c_int32, i64, vp, vp,
                                       ctypes.c_float, ctypes.c_float, i32, ctypes.POINTER(Plan), vp]
        lib.rmsnorm_qk_fwd.restype = i32
        lib.rmsnorm_qk_plan_for.argtypes = [vp, vp, i64, i64, i64, ctypes.c_int32, ctypes.c_int32, i64, vp, vp,
                                            i32, ctypes.POINTER(Plan)]
        lib.rmsnorm_qk_plan_for.restype = i32
        lib.rmsnorm_fwd_mxfp8.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, ctypes.c_float, ctypes.c_float, i32,
                                          ctypes.POINTER(Plan), vp]
        lib.rmsnorm_fwd_mxfp8.restype = i32
        lib.rmsnorm_mxfp8_plan_for.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, ctypes.POINTER(Plan)]
        lib.rmsnorm_mxfp8_plan_for.restype = i32
        lib.rmsnorm_fwd_nvfp4.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, ctypes.c_float, ctypes.c_float,
                                          ctypes.c_float, i32, ctypes.POINTER(Plan), vp]
        lib.rmsnorm_fwd_nvfp4.restype = i32
        lib.rmsnorm_nvfp4_plan_for.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, ctypes.POINTER(Plan)]
        lib.rmsnorm_nvfp4_plan_for.restype = i32
        lib.layernorm_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, ctypes.c_float, i32,
                                      ctypes.POINTER(Plan), vp]
        lib.layernorm_fwd.restype = i32
        lib.layernorm_plan_for.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, ctypes.POINTER(Plan)]
        lib.layernorm_plan_for.restype = i32
        lib.rmsnorm_plan.argtypes = [i64, i64, i32, i32, i32, i32, ctypes.POINTER(Plan)]
        lib.rmsnorm_plan.restype = i32
        lib.rmsnorm_plan_ex.argtypes = [i64, i64, i32, i32, i32, i32, i32, ctypes.POINTER(Plan)]
        lib.rmsnorm_plan_ex.restype = i32
        lib.rmsnorm_plan_for.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, ctypes.POINTER(Plan)]
        lib.rmsnorm_plan_for.restype = i32
        lib.rmsnorm_regime.argtypes = [i64, i64, i32]
        lib.rmsnorm_regime.restype = i32
        lib.rmsnorm_max_hidden.argtypes = [i32]
        lib.rmsnorm_max_hidden.restype = i64
        lib.rmsnorm_reg_max_chunks.argtypes = []
        lib.rmsnorm_reg_max_chunks.restype = i32
        lib.rmsnorm_tma_wait_test.argtypes = fwd_args + [ctypes.POINTER(Plan), ctypes.c_uint64, i32, vp]
        lib.rmsnorm_tma_wait_test.restype = i32
        lib.rmsnorm_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.rmsnorm_wait_timeouts.restype = i32
        lib.rmsnorm_fwd_host.argtypes = fwd_args + [vp, ctypes.c_uint64, i64, vp]
        lib.rmsnorm_fwd_host.restype = i32
        lib.rmsnorm_host_workspace_bytes.argtypes = [i64, i64, i32, i32]
        lib.rmsnorm_host_workspace_bytes.restype = i64
        lib.rmsnorm_fwd_host_static.argtypes = fwd_args + [vp]
        lib.rmsnorm_fwd_host_static.restype = i32
        lib.rmsnorm_strerror.argtypes = [i32]
        lib.rmsnorm_strerror.restype = ctypes.c_char_p
        lib.rmsnorm_build_info.argtypes = []
        lib.rmsnorm_build_info.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != RMSNORM_OK:
        raise RmsNormError(status, where)


def rmsnorm_fwd(x, residual, w, y, residual_out, rows, hidden, eps, dtype, stream=0):
    _check(load().rmsnorm_fwd(x, residual, w, y, residual_out, rows, hidden, eps, dtype, stream),
           "rmsnorm_fwd")


def rmsnorm_fwd_status(x, residual, w, y, residual_out, rows, hidden, eps, dtype, stream=0) -> int:
    """rmsnorm_fwd returning the raw status instead of raising."""
    return load().rmsnorm_fwd(x, residual, w, y, residual_out, rows, hidden, eps, dtype, stream)


def rmsnorm_fwd_plan(x, residual, w, y, residual_out, rows, hidden, eps, dtype, plan: Plan, stream=0):
    _check(load().rmsnorm_fwd_plan(x, residual, w, y, residual_out, rows, hidden, eps, dtype,
                                   ctypes.byref(plan), stream), "rmsnorm_fwd_plan")


def rmsnorm_fwd_plan_status(x, residual, w, y, residual_out, rows, hidden, eps, dtype, plan, stream=0):
    return load().rmsnorm_fwd_plan(x, residual, w, y, residual_out, rows, hidden, eps, dtype,
                                   ctypes.byref(plan) if plan is not None else None, stream)


def _plan_ref(plan):
    return None if plan is None else ctypes.byref(plan)


def rmsnorm_fwd_ex(x, residual, w, y, residual_out, rows, hidden, eps, weight_bias, dtype, plan=None,
                   stream=0):
    _check(load().rmsnorm_fwd_ex(x, residual, w, y, residual_out, rows, hidden, eps, weight_bias, dtype,
                                 _plan_ref(plan), stream), "rmsnorm_fwd_ex")


def rmsnorm_fwd_ex_status(x, residual, w, y, residual_out, rows, hidden, eps, weight_bias, dtype, plan=None,
                          stream=0) -> int:
    return load().rmsnorm_fwd_ex(x, residual, w, y, residual_out, rows, hidden, eps, weight_bias, dtype,
                                 _plan_ref(plan), stream)


def rmsnorm_fwd_cast(x, residual, w, y, residual_out, rows, hidden, eps, dtype, plan=None, stream=0):
    _check(load().rmsnorm_fwd_cast(x, residual, w, y, residual_out, rows, hidden, eps, dtype, _plan_ref(plan),
                                   stream), "rmsnorm_fwd_cast")


def rmsnorm_fwd_cast_status(x, residual, w, y, residual_out, rows, hidden, eps, dtype, plan=None, stream=0) -> int:
    return load().rmsnorm_fwd_cast(x, residual, w, y, residual_out, rows, hidden, eps, dtype, _plan_ref(plan),
                                   stream)


def rmsnorm_qk_fwd(x, y, tokens, x_token_stride, y_token_stride, q_heads, k_heads, head_dim, q_w, k_w,
                   weight_bias, eps, dtype, plan=None, stream=0):
    _check(rmsnorm_qk_fwd_status(x, y, tokens, x_token_stride, y_token_stride, q_heads, k_heads, head_dim,
                                 q_w, k_w, weight_bias, eps, dtype, plan, stream), "rmsnorm_qk_fwd")


def rmsnorm_qk_fwd_status(x, y, tokens, x_token_stride, y_token_stride, q_heads, k_heads, head_dim, q_w, k_w,
                          weight_bias, eps, dtype, plan=None, stream=0) -> int:
    return load().rmsnorm_qk_fwd(x, y, tokens, x_token_stride, y_token_stride, q_heads, k_heads, head_dim,
                                 q_w, k_w, weight_bias, eps, dtype, _plan_ref(plan), stream)


def rmsnorm_qk_plan_for(x, y, tokens, x_token_stride, y_token_stride, q_heads, k_heads, head_dim, q_w, k_w,
                        dtype) -> Plan:
    p = Plan()
    _check(load().rmsnorm_qk_plan_for(x, y, tokens, x_token_stride, y_token_stride, q_heads, k_heads,
                                      head_dim, q_w, k_w, dtype, ctypes.byref(p)), "rmsnorm_qk_plan_for")
    return p


def rmsnorm_fwd_mxfp8(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias, dtype,
                      plan=None, stream=0):
    _check(rmsnorm_fwd_mxfp8_status(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias,
                                    dtype, plan, stream), "rmsnorm_fwd_mxfp8")


def rmsnorm_fwd_mxfp8_status(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias, dtype,
                             plan=None, stream=0) -> int:
    return load().rmsnorm_fwd_mxfp8(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias,
                                    dtype, _plan_ref(plan), stream)


def rmsnorm_mxfp8_plan_for(x, residual, w, codes, scales, residual_out, rows, hidden, dtype) -> Plan:
    p = Plan()
    _check(load().rmsnorm_mxfp8_plan_for(x, residual, w, codes, scales, residual_out, rows, hidden, dtype,
                                         ctypes.byref(p)), "rmsnorm_mxfp8_plan_for")
    return p


def rmsnorm_fwd_nvfp4(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias, tensor_scale,
                      dtype, plan=None, stream=0):
    _check(rmsnorm_fwd_nvfp4_status(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias,
                                    tensor_scale, dtype, plan, stream), "rmsnorm_fwd_nvfp4")


def rmsnorm_fwd_nvfp4_status(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias,
                             tensor_scale, dtype, plan=None, stream=0) -> int:
    return load().rmsnorm_fwd_nvfp4(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias,
                                    tensor_scale, dtype, _plan_ref(plan), stream)


def rmsnorm_nvfp4_plan_for(x, residual, w, codes, scales, residual_out, rows, hidden, dtype) -> Plan:
    p = Plan()
    _check(load().rmsnorm_nvfp4_plan_for(x, residual, w, codes, scales, residual_out, rows, hidden, dtype,
                                         ctypes.byref(p)), "rmsnorm_nvfp4_plan_for")
    return p


def layernorm_fwd(x, residual, w, b, y, residual_out, rows, hidden, eps, dtype, plan=None, stream=0):
    _check(layernorm_fwd_status(x, residual, w, b, y, residual_out, rows, hidden, eps, dtype, plan, stream),
           "layernorm_fwd")


def layernorm_fwd_status(x, residual, w, b, y, residual_out, rows, hidden, eps, dtype, plan=None,
                         stream=0) -> int:
    return load().layernorm_fwd(x, residual, w, b, y, residual_out, rows, hidden, eps, dtype, _plan_ref(plan),
                                stream)


def layernorm_plan_for(x, residual, w, b, y, residual_out, rows, hidden, dtype) -> Plan:
    p = Plan()
    _check(load().layernorm_plan_for(x, residual, w, b, y, residual_out, rows, hidden, dtype, ctypes.byref(p)),
           "layernorm_plan_for")
    return p


def rmsnorm_plan(rows, hidden, dtype, vec_ok, sm_count, blocks_per_sm) -> Plan:
    p = Plan()
    _check(load().rmsnorm_plan(rows, hidden, dtype, int(vec_ok), sm_count, blocks_per_sm,
                               ctypes.byref(p)), "rmsnorm_plan")
    return p


def rmsnorm_plan_ex(rows, hidden, dtype, vec_ok, has_residual, sm_count, blocks_per_sm) -> Plan:
    p = Plan()
    _check(load().rmsnorm_plan_ex(rows, hidden, dtype, int(vec_ok), int(has_residual), sm_count, blocks_per_sm,
                                  ctypes.byref(p)), "rmsnorm_plan_ex")
    return p


def rmsnorm_plan_for(x, residual, w, y, residual_out, rows, hidden, dtype) -> Plan:
    p = Plan()
    _check(load().rmsnorm_plan_for(x, residual, w, y, residual_out, rows, hidden, dtype,
                                   ctypes.byref(p)), "rmsnorm_plan_for")
    return p


def rmsnorm_regime(rows, hidden, dtype) -> int:
    """The RMSNORM_REGIME_* rmsnorm_fwd runs on the current device for aligned
    contiguous tensors with a weight and no residual."""
    st = int(load().rmsnorm_regime(rows, hidden, dtype))
    if st < 0:
        raise RmsNormError(st, "rmsnorm_regime")
    return st


def rmsnorm_regime_status(rows, hidden, dtype) -> int:
    """rmsnorm_regime's raw return value: a regime (>= 0) or a negative status."""
    return int(load().rmsnorm_regime(rows, hidden, dtype))


def rmsnorm_fwd_host(x, residual, w, y, residual_out, rows, hidden, eps, dtype, workspace, workspace_bytes,
                     chunk_rows, stream=0):
    """The op on HOST pointers, streamed through the device in chunks (see
    the header); asynchronous on ``stream``."""
    _check(load().rmsnorm_fwd_host(x, residual, w, y, residual_out, rows, hidden, eps, dtype, workspace,
                                   workspace_bytes, chunk_rows, stream), "rmsnorm_fwd_host")


def rmsnorm_fwd_host_status(x, residual, w, y, residual_out, rows, hidden, eps, dtype, workspace,
                            workspace_bytes, chunk_rows, stream=0) -> int:
    return load().rmsnorm_fwd_host(x, residual, w, y, residual_out, rows, hidden, eps, dtype, workspace,
                                   workspace_bytes, chunk_rows, stream)


def rmsnorm_fwd_host_static(x, residual, w, y, residual_out, rows, hidden, eps, dtype, stream=0):
    """rmsnorm_fwd_host with the library's own device scratch (no workspace)."""
    _check(load().rmsnorm_fwd_host_static(x, residual, w, y, residual_out, rows, hidden, eps, dtype, stream),
           "rmsnorm_fwd_host_static")


def rmsnorm_host_workspace_bytes(chunk_rows, hidden, dtype, has_residual) -> int:
    n = int(load().rmsnorm_host_workspace_bytes(chunk_rows, hidden, dtype, int(has_residual)))
    if n < 0:
        raise RmsNormError(n, "rmsnorm_host_workspace_bytes")
    return n


def rmsnorm_max_hidden(dtype) -> int:
    return int(load().rmsnorm_max_hidden(dtype))


def rmsnorm_reg_max_chunks() -> int:
    return int(load().rmsnorm_reg_max_chunks())


def rmsnorm_strerror(status) -> str:
    return load().rmsnorm_strerror(int(status)).decode()


def rmsnorm_build_info() -> str:
    return load().rmsnorm_build_info().decode()


def rmsnorm_tma_wait_test_status(x, residual, w, y, residual_out, rows, hidden, eps, dtype, plan, wait_limit_ns,
                                 withhold_release, stream=0) -> int:
    """The bulk-copy kernel's bounded-wait test hook (see the header); returns the status."""
    return load().rmsnorm_tma_wait_test(x, residual, w, y, residual_out, rows, hidden, eps, dtype, _plan_ref(plan),
                                        wait_limit_ns, withhold_release, stream)


def rmsnorm_wait_timeouts() -> int:
    """Blocks of the bulk-copy kernel on the current device whose bounded
    waits ran out since the library was loaded (a blocking read)."""
    n = ctypes.c_uint32(0)
    _check(load().rmsnorm_wait_timeouts(ctypes.byref(n)), "rmsnorm_wait_timeouts")
    return int(n.value)
