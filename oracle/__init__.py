"""Oracle: a plain fp64 CPU reference for the fused row-wise RMSNorm.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
and the benchmark's CPU-baseline / reference legs may import this package.
It shares no code with the CUDA library and never imports it.

The arithmetic lives in ``rmsnorm_oracle.c`` (plain C, binary64, built with
``-O2 -ffp-contract=off`` and no fast-math).  This module only compiles that
file with gcc, loads it with ctypes and passes numpy buffers to it.  Rows are
independent, so ``threads > 1`` splits the row range into contiguous blocks and
runs one C call per block on a thread pool (ctypes releases the GIL for the
call); the per-row arithmetic is unchanged by that split.

What it computes follows the RMSNorm definition of "Building a GPU compiler
from scratch: from PyTorch to CUDA via multi-level IR (Emmy)" (running example
and section "Tensor IR"); the C file lists the readings taken where the pages
are silent.

Data convention: bf16 tensors are numpy ``uint16`` arrays of raw bf16 bits;
fp32 tensors are numpy ``float32`` arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_rmsnorm.so")

DTYPES = {"f32": 0, "bf16": 1}
_NP_TYPE = {"f32": np.float32, "bf16": np.uint16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build`` with gcc and return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
               "-Wall", "-Wextra", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i64 = ctypes.c_void_p, ctypes.c_int64
            lib.oracle_rmsnorm_rows.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                                ctypes.c_float, ctypes.c_float, ctypes.c_int]
            lib.oracle_rmsnorm_rows.restype = ctypes.c_int
            lib.oracle_rmsnorm_cast_rows.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                                     ctypes.c_float, ctypes.c_int]
            lib.oracle_rmsnorm_cast_rows.restype = ctypes.c_int
            lib.oracle_layernorm_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                                  ctypes.c_float, ctypes.c_int]
            lib.oracle_layernorm_rows.restype = ctypes.c_int
            lib.oracle_rmsnorm_mxfp8_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                                      ctypes.c_float, ctypes.c_float, ctypes.c_int]
            lib.oracle_rmsnorm_mxfp8_rows.restype = ctypes.c_int
            lib.oracle_rmsnorm_nvfp4_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                                      ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                      ctypes.c_int]
            lib.oracle_rmsnorm_nvfp4_rows.restype = ctypes.c_int
            lib.oracle_e2m1_from_double.argtypes = [vp, vp, i64]
            lib.oracle_e2m1_from_double.restype = None
            lib.oracle_double_from_e2m1.argtypes = [vp, vp, i64]
            lib.oracle_double_from_e2m1.restype = None
            lib.oracle_e4m3_from_double.argtypes = [vp, vp, i64]
            lib.oracle_e4m3_from_double.restype = None
            lib.oracle_double_from_e4m3.argtypes = [vp, vp, i64]
            lib.oracle_double_from_e4m3.restype = None
            lib.oracle_bf16_from_double.argtypes = [vp, vp, i64]
            lib.oracle_bf16_from_double.restype = None
            lib.oracle_double_from_bf16.argtypes = [vp, vp, i64]
            lib.oracle_double_from_bf16.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(a, name, dtype, shape):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != _NP_TYPE[dtype]:
        raise TypeError(f"{name}: expected {_NP_TYPE[dtype].__name__} for dtype {dtype}, got {a.dtype}")
    if a.shape != shape:
        raise ValueError(f"{name}: expected shape {shape}, got {a.shape}")
    return a


def rmsnorm(x, w=None, residual=None, eps: float = 1e-6, dtype: str = "bf16",
            want_exact: bool = False, threads: int = 1, weight_bias: float = 0.0):
    """Reference RMSNorm of every row of ``x`` ([rows, hidden]).

    Returns ``(y, residual_out, y_exact)``: ``y`` in the I/O type,
    ``residual_out`` (= the rounded ``x + residual``) or None, and the fp64
    value of ``y`` before its final rounding, or None unless ``want_exact``.
    ``weight_bias`` is added to every weight element (float value).
    """
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    x = np.ascontiguousarray(x)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [rows, hidden]")
    rows, hidden = x.shape
    x = _check(x, "x", dtype, (rows, hidden))
    residual = _check(residual, "residual", dtype, (rows, hidden))
    w = _check(w, "w", dtype, (hidden,))

    y = np.empty((rows, hidden), dtype=_NP_TYPE[dtype])
    res_out = None if residual is None else np.empty((rows, hidden), dtype=_NP_TYPE[dtype])
    y64 = np.empty((rows, hidden), dtype=np.float64) if want_exact else None
    if rows == 0 or hidden == 0:
        return y, res_out, y64

    lib = _load()
    args = (_ptr(x), _ptr(residual), _ptr(w), _ptr(y), _ptr(y64), _ptr(res_out))

    def run(lo, hi):
        rc = lib.oracle_rmsnorm_rows(*args, lo, hi, hidden, float(eps), float(weight_bias), DTYPES[dtype])
        if rc != 0:
            raise ValueError("oracle rejected its arguments")

    threads = max(1, min(int(threads), rows))
    if threads == 1:
        run(0, rows)
    else:
        bounds = np.linspace(0, rows, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])), range(threads)))
    return y, res_out, y64


def rmsnorm_cast(x, w=None, residual=None, eps: float = 1e-6, dtype: str = "bf16", threads: int = 1):
    """Reference RMSNorm in the op-by-op cast order (see the C file): the
    normalised value is rounded to the I/O type before the weight multiply.

    Returns ``(y, residual_out, n_exact)``: ``y`` in the I/O type, the rounded
    residual sum or None, and the fp64 normalised values h * r before their
    rounding.
    """
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    x = np.ascontiguousarray(x)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [rows, hidden]")
    rows, hidden = x.shape
    x = _check(x, "x", dtype, (rows, hidden))
    residual = _check(residual, "residual", dtype, (rows, hidden))
    w = _check(w, "w", dtype, (hidden,))
    y = np.empty((rows, hidden), dtype=_NP_TYPE[dtype])
    res_out = None if residual is None else np.empty((rows, hidden), dtype=_NP_TYPE[dtype])
    n64 = np.empty((rows, hidden), dtype=np.float64)
    if rows == 0 or hidden == 0:
        return y, res_out, n64
    lib = _load()
    args = (_ptr(x), _ptr(residual), _ptr(w), _ptr(y), _ptr(n64), _ptr(res_out))

    def run(lo, hi):
        if lib.oracle_rmsnorm_cast_rows(*args, lo, hi, hidden, float(eps), DTYPES[dtype]) != 0:
            raise ValueError("oracle rejected its arguments")

    threads = max(1, min(int(threads), rows))
    if threads == 1:
        run(0, rows)
    else:
        bounds = np.linspace(0, rows, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])), range(threads)))
    return y, res_out, n64


def layernorm(x, w=None, b=None, residual=None, eps: float = 1e-5, dtype: str = "bf16",
              want_exact: bool = False, threads: int = 1):
    """Reference LayerNorm of every row of ``x`` ([rows, hidden]) ("GPT-2 on the
    GPU", section "The Whole Model as One Kernel").

    Returns ``(y, residual_out, n_exact, y_exact)``; the last two (fp64 values
    of the normalised row and of y before rounding) only with ``want_exact``.
    """
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    x = np.ascontiguousarray(x)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [rows, hidden]")
    rows, hidden = x.shape
    x = _check(x, "x", dtype, (rows, hidden))
    residual = _check(residual, "residual", dtype, (rows, hidden))
    w = _check(w, "w", dtype, (hidden,))
    b = _check(b, "b", dtype, (hidden,))
    y = np.empty((rows, hidden), dtype=_NP_TYPE[dtype])
    res_out = None if residual is None else np.empty((rows, hidden), dtype=_NP_TYPE[dtype])
    n64 = np.empty((rows, hidden), dtype=np.float64) if want_exact else None
    y64 = np.empty((rows, hidden), dtype=np.float64) if want_exact else None
    if rows == 0 or hidden == 0:
        return y, res_out, n64, y64
    lib = _load()
    args = (_ptr(x), _ptr(residual), _ptr(w), _ptr(b), _ptr(y), _ptr(n64), _ptr(y64), _ptr(res_out))

    def run(lo, hi):
        rc = lib.oracle_layernorm_rows(*args, lo, hi, hidden, float(eps), DTYPES[dtype])
        if rc != 0:
            raise ValueError("oracle rejected its arguments")

    threads = max(1, min(int(threads), rows))
    if threads == 1:
        run(0, rows)
    else:
        bounds = np.linspace(0, rows, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])), range(threads)))
    return y, res_out, n64, y64


def rmsnorm_mxfp8(x, w=None, residual=None, eps: float = 1e-6, dtype: str = "bf16", weight_bias: float = 0.0,
                  threads: int = 1):
    """Reference RMSNorm with MXFP8 output (E4M3 codes, one E8M0 scale per 32
    elements of a row; see the C file for the exact rule).

    Returns ``(codes, scales, residual_out, v_exact)``: uint8 codes [rows,
    hidden], uint8 scales [rows, hidden/32], the rounded residual sum or None,
    and the op's fp64 values before quantisation.
    """
    x = np.ascontiguousarray(x)
    rows, hidden = x.shape
    x = _check(x, "x", dtype, (rows, hidden))
    residual = _check(residual, "residual", dtype, (rows, hidden))
    w = _check(w, "w", dtype, (hidden,))
    if hidden % 32:
        raise ValueError("hidden must be a multiple of 32")
    codes = np.empty((rows, hidden), dtype=np.uint8)
    scales = np.empty((rows, hidden // 32), dtype=np.uint8)
    res_out = None if residual is None else np.empty((rows, hidden), dtype=_NP_TYPE[dtype])
    v64 = np.empty((rows, hidden), dtype=np.float64)
    if rows == 0:
        return codes, scales, res_out, v64
    lib = _load()
    args = (_ptr(x), _ptr(residual), _ptr(w), _ptr(codes), _ptr(scales), _ptr(v64), _ptr(res_out))

    def run(lo, hi):
        rc = lib.oracle_rmsnorm_mxfp8_rows(*args, lo, hi, hidden, float(eps), float(weight_bias), DTYPES[dtype])
        if rc != 0:
            raise ValueError("oracle rejected its arguments")

    threads = max(1, min(int(threads), rows))
    if threads == 1:
        run(0, rows)
    else:
        bounds = np.linspace(0, rows, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])), range(threads)))
    return codes, scales, res_out, v64


def rmsnorm_nvfp4(x, w=None, residual=None, eps: float = 1e-6, dtype: str = "bf16", weight_bias: float = 0.0,
                  tensor_scale: float = 1.0, threads: int = 1):
    """Reference RMSNorm with NVFP4 output (E2M1 codes packed two a byte, one
    E4M3 scale per 16 elements, per-tensor scale ``tensor_scale``; see the C
    file).  Returns ``(codes [rows, hidden/2], scales [rows, hidden/16],
    residual_out, v_exact)``."""
    x = np.ascontiguousarray(x)
    rows, hidden = x.shape
    x = _check(x, "x", dtype, (rows, hidden))
    residual = _check(residual, "residual", dtype, (rows, hidden))
    w = _check(w, "w", dtype, (hidden,))
    if hidden % 16:
        raise ValueError("hidden must be a multiple of 16")
    codes = np.empty((rows, hidden // 2), dtype=np.uint8)
    scales = np.empty((rows, hidden // 16), dtype=np.uint8)
    res_out = None if residual is None else np.empty((rows, hidden), dtype=_NP_TYPE[dtype])
    v64 = np.empty((rows, hidden), dtype=np.float64)
    if rows == 0:
        return codes, scales, res_out, v64
    lib = _load()
    args = (_ptr(x), _ptr(residual), _ptr(w), _ptr(codes), _ptr(scales), _ptr(v64), _ptr(res_out))

    def run(lo, hi):
        rc = lib.oracle_rmsnorm_nvfp4_rows(*args, lo, hi, hidden, float(eps), float(weight_bias),
                                           float(tensor_scale), DTYPES[dtype])
        if rc != 0:
            raise ValueError("oracle rejected its arguments")

    threads = max(1, min(int(threads), rows))
    if threads == 1:
        run(0, rows)
    else:
        bounds = np.linspace(0, rows, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])), range(threads)))
    return codes, scales, res_out, v64


def e2m1_from_double(v) -> np.ndarray:
    """Round fp64 values to 4-bit E2M1 codes (nearest-even, saturated at 6)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e2m1_from_double(_ptr(v), _ptr(out), v.size)
    return out


def double_from_e2m1(c) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_double_from_e2m1(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_from_double(v) -> np.ndarray:
    """Round fp64 values to E4M3 codes (nearest-even, saturated at 448)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_from_double(_ptr(v), _ptr(out), v.size)
    return out


def double_from_e4m3(c) -> np.ndarray:
    """Decode E4M3 codes."""
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_double_from_e4m3(_ptr(c), _ptr(out), c.size)
    return out


def rmsnorm_qk(x, q_heads: int, k_heads: int, head_dim: int, q_w=None, k_w=None, eps: float = 1e-6,
               dtype: str = "bf16", weight_bias: float = 0.0, threads: int = 1):
    """Reference per-head RMSNorm of the query and key heads of packed token rows.

    ``x`` is [tokens, stride] with stride >= (q_heads + k_heads) * head_dim:
    query head j of a token occupies columns [j*head_dim, (j+1)*head_dim),
    key head j the columns after the query heads.  Each head is one row of
    the op above, with ``q_w`` for query heads and ``k_w`` for key heads
    ("CuTeDSL at Perplexity", section "QK Norm").  Returns ``(q_y, k_y)`` of
    shapes [tokens, q_heads, head_dim] and [tokens, k_heads, head_dim]; the
    columns past the key heads are not part of the op.
    """
    x = np.ascontiguousarray(x)
    tokens = x.shape[0]
    q_cols = q_heads * head_dim
    k_cols = k_heads * head_dim
    q_rows = x[:, :q_cols].reshape(tokens * q_heads, head_dim)
    k_rows = x[:, q_cols:q_cols + k_cols].reshape(tokens * k_heads, head_dim)
    qy = rmsnorm(q_rows, w=q_w, eps=eps, dtype=dtype, threads=threads, weight_bias=weight_bias)[0]
    ky = rmsnorm(k_rows, w=k_w, eps=eps, dtype=dtype, threads=threads, weight_bias=weight_bias)[0]
    return qy.reshape(tokens, q_heads, head_dim), ky.reshape(tokens, k_heads, head_dim)


def bf16_from_double(v) -> np.ndarray:
    """Round fp64 values to bf16 bits (round to nearest, ties to even)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_from_double(_ptr(v), _ptr(out), v.size)
    return out


def double_from_bf16(bits) -> np.ndarray:
    """Decode bf16 bits to fp64 values."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_double_from_bf16(_ptr(bits), _ptr(out), bits.size)
    return out
