"""Torch-facing call of the fused RMSNorm: tensors in, the C ABI underneath.

``rms_norm`` only checks shapes, allocates missing outputs with torch (the
caller's allocator, on the tensors' device) and passes raw pointers and the
current stream to ``rmsnorm_fwd``.  CPU tensors are refused: there is no
fallback path.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _native as N

_CODES = {torch.bfloat16: N.RMSNORM_BF16, torch.float32: N.RMSNORM_F32}


def dtype_code(dtype: torch.dtype) -> int:
    try:
        return _CODES[dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {dtype}: bf16 or fp32 only") from None


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_tensor(t, name, x):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if t.device != x.device:
        raise ValueError(f"{name} is on {t.device}, x on {x.device}")
    if t.dtype != x.dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, x has {x.dtype}: one I/O type for all tensors")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def rms_norm(x: torch.Tensor, w: Optional[torch.Tensor] = None, residual: Optional[torch.Tensor] = None,
             eps: float = 1e-6, out: Optional[torch.Tensor] = None,
             residual_out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
             plan: Optional[N.Plan] = None, weight_bias: float = 0.0, cast_before_weight: bool = False):
    """y = x * rsqrt(mean(x^2) + eps) * (w + weight_bias) over the last dimension.

    With ``residual``: h = x + residual (rounded to the I/O type) is written to
    ``residual_out`` and normalised; returns ``(y, residual_out)``.  Without:
    returns ``y``.  ``plan`` forces a launch plan (see ``rmsnorm_fwd_plan``).
    ``weight_bias`` = 1 gives the (1 + w) weight form.  ``cast_before_weight``
    rounds the normalised value to the I/O type before the weight multiply
    (``rmsnorm_fwd_cast``, the eager op-by-op order; no weight bias).
    """
    if x.dim() < 1:
        raise ValueError("x must have at least one dimension")
    _check_tensor(x, "x", x)
    code = dtype_code(x.dtype)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    for name, t in (("residual", residual), ("out", out), ("residual_out", residual_out)):
        if t is not None and t.shape != x.shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, x has {tuple(x.shape)}")
    if w is not None and tuple(w.shape) != (hidden,):
        raise ValueError(f"w must have shape ({hidden},), got {tuple(w.shape)}")
    y = torch.empty_like(x) if out is None else out
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    for name, t in (("w", w), ("residual", residual), ("out", y), ("residual_out", residual_out)):
        _check_tensor(t, name, x)
    with torch.cuda.device(x.device):
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        args = (_ptr(x), _ptr(residual), _ptr(w), _ptr(y), _ptr(residual_out), rows, hidden,
                float(eps))
        if cast_before_weight:
            if weight_bias:
                raise ValueError("cast_before_weight takes no weight_bias")
            N.rmsnorm_fwd_cast(*args, code, plan, s.cuda_stream)
        elif weight_bias:
            N.rmsnorm_fwd_ex(*args, float(weight_bias), code, plan, s.cuda_stream)
        elif plan is None:
            N.rmsnorm_fwd(*args, code, s.cuda_stream)
        else:
            N.rmsnorm_fwd_plan(*args, code, plan, s.cuda_stream)
    return (y, residual_out) if residual is not None else y


def rms_norm_host(x: torch.Tensor, w: Optional[torch.Tensor] = None, residual: Optional[torch.Tensor] = None,
                  eps: float = 1e-6, out: Optional[torch.Tensor] = None, residual_out: Optional[torch.Tensor] = None,
                  chunk_rows: int = 4096, workspace: Optional[torch.Tensor] = None,
                  device: Optional[torch.device] = None, stream: Optional[torch.cuda.Stream] = None):
    """``rms_norm`` on CPU tensors, streamed through a GPU in chunks of
    ``chunk_rows`` rows (``rmsnorm_fwd_host``): uploads, launches and
    read-backs overlap when the tensors are in pinned memory.  ``workspace``
    is a CUDA uint8 tensor of at least ``rmsnorm_host_workspace_bytes(...)``
    bytes
    (allocated on ``device`` when not given).  Returns after the work is
    queued on ``stream``: synchronise it before reading the outputs."""
    if x.dim() < 1:
        raise ValueError("x must have at least one dimension")
    code = dtype_code(x.dtype)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    y = torch.empty_like(x) if out is None else out
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    for name, t in (("x", x), ("w", w), ("residual", residual), ("out", y), ("residual_out", residual_out)):
        if t is None:
            continue
        if t.is_cuda:
            raise ValueError(f"{name} must be a CPU tensor (use rms_norm for device tensors)")
        if t.dtype != x.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous with dtype {x.dtype}")
        if name != "w" and t.shape != x.shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, x has {tuple(x.shape)}")
    if w is not None and tuple(w.shape) != (hidden,):
        raise ValueError(f"w must have shape ({hidden},), got {tuple(w.shape)}")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    need = N.rmsnorm_host_workspace_bytes(chunk_rows, hidden, code, residual is not None)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    with torch.cuda.device(workspace.device):
        s = stream if stream is not None else torch.cuda.current_stream(workspace.device)
        N.rmsnorm_fwd_host(_ptr(x), _ptr(residual), _ptr(w), _ptr(y), _ptr(residual_out), rows, hidden,
                           float(eps), code, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                           chunk_rows, s.cuda_stream)
    return (y, residual_out) if residual is not None else y


def _token_view(t: torch.Tensor, name: str):
    """(tokens, token_stride) of a [tokens, width] tensor with a contiguous last dimension."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D [tokens, width] tensor")
    if t.stride(1) != 1 and t.shape[1] > 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")
    return t.shape[0], t.stride(0), t


def qk_norm(qkv: torch.Tensor, q_heads: int, k_heads: int, head_dim: int, q_w: Optional[torch.Tensor] = None,
            k_w: Optional[torch.Tensor] = None, eps: float = 1e-6, weight_bias: float = 0.0,
            out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
            plan: Optional[N.Plan] = None) -> torch.Tensor:
    """Per-head RMSNorm of the query and key heads of packed token rows in one launch.

    ``qkv`` is [tokens, width] (last dimension contiguous, token rows evenly
    strided, e.g. a view of a fused projection) holding q_heads query heads, then
    k_heads key heads of head_dim elements, then anything else (value heads),
    which is left alone.  Query heads take ``q_w``, key heads ``k_w``.  The
    result goes to ``out`` (same layout; pass ``out=qkv`` to normalise in
    place) or to a new tensor whose other columns are copied from ``qkv``.
    """
    _check_tensor(qkv, "qkv", qkv)
    code = dtype_code(qkv.dtype)
    tokens, xs, rows = _token_view(qkv, "qkv")
    if out is None:
        out = qkv.clone()
    if out.shape != qkv.shape:
        raise ValueError("out must have the shape of qkv")
    _, ys, _ = _token_view(out, "out")
    for name, t in (("q_w", q_w), ("k_w", k_w)):
        if t is not None:
            _check_tensor(t, name, qkv)
            if tuple(t.shape) != (head_dim,):
                raise ValueError(f"{name} must have shape ({head_dim},)")
    if out.device != qkv.device or out.dtype != qkv.dtype:
        raise ValueError("out must match qkv's device and dtype")
    with torch.cuda.device(qkv.device):
        s = stream if stream is not None else torch.cuda.current_stream(qkv.device)
        N.rmsnorm_qk_fwd(_ptr(qkv), _ptr(out), tokens, xs, ys, int(q_heads), int(k_heads), int(head_dim),
                         _ptr(q_w), _ptr(k_w), float(weight_bias), float(eps), code, plan, s.cuda_stream)
    return out


def qk_plan_for(qkv: torch.Tensor, q_heads: int, k_heads: int, head_dim: int, q_w=None, k_w=None,
                out=None) -> N.Plan:
    """The plan ``qk_norm`` would launch for these tensors."""
    tokens, xs, _ = _token_view(qkv, "qkv")
    y = qkv if out is None else out
    _, ys, _ = _token_view(y, "out")
    with torch.cuda.device(qkv.device):
        return N.rmsnorm_qk_plan_for(_ptr(qkv), _ptr(y), tokens, xs, ys, int(q_heads), int(k_heads),
                                     int(head_dim), _ptr(q_w), _ptr(k_w), dtype_code(qkv.dtype))


def plan_for(x: torch.Tensor, w=None, residual=None, out=None, residual_out=None) -> N.Plan:
    """The plan ``rms_norm`` would launch for these tensors."""
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    y = out if out is not None else x
    ro = residual_out if residual_out is not None else residual
    with torch.cuda.device(x.device):
        return N.rmsnorm_plan_for(_ptr(x), _ptr(residual), _ptr(w), _ptr(y), _ptr(ro), rows, hidden,
                                  dtype_code(x.dtype))


def layer_norm(x: torch.Tensor, w: Optional[torch.Tensor] = None, b: Optional[torch.Tensor] = None,
               residual: Optional[torch.Tensor] = None, eps: float = 1e-5, out: Optional[torch.Tensor] = None,
               residual_out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
               plan: Optional[N.Plan] = None):
    """y = (h - mean(h)) / sqrt(var(h) + eps) * w + b over the last dimension
    (h = x, or x + residual written to ``residual_out``).  Returns y, or
    (y, residual_out) with a residual."""
    _check_tensor(x, "x", x)
    code = dtype_code(x.dtype)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    for name, t in (("residual", residual), ("out", out), ("residual_out", residual_out)):
        if t is not None and t.shape != x.shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, x has {tuple(x.shape)}")
    for name, t in (("w", w), ("b", b)):
        if t is not None and tuple(t.shape) != (hidden,):
            raise ValueError(f"{name} must have shape ({hidden},)")
    y = torch.empty_like(x) if out is None else out
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    for name, t in (("w", w), ("b", b), ("residual", residual), ("out", y), ("residual_out", residual_out)):
        _check_tensor(t, name, x)
    with torch.cuda.device(x.device):
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        N.layernorm_fwd(_ptr(x), _ptr(residual), _ptr(w), _ptr(b), _ptr(y), _ptr(residual_out), rows, hidden,
                        float(eps), code, plan, s.cuda_stream)
    return (y, residual_out) if residual is not None else y


def layer_norm_plan_for(x, w=None, b=None, residual=None, out=None, residual_out=None) -> N.Plan:
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    y = out if out is not None else x
    ro = residual_out if residual_out is not None else residual
    with torch.cuda.device(x.device):
        return N.layernorm_plan_for(_ptr(x), _ptr(residual), _ptr(w), _ptr(b), _ptr(y), _ptr(ro), rows, hidden,
                                    dtype_code(x.dtype))


def rms_norm_mxfp8(x: torch.Tensor, w: Optional[torch.Tensor] = None, residual: Optional[torch.Tensor] = None,
                   eps: float = 1e-6, weight_bias: float = 0.0, codes: Optional[torch.Tensor] = None,
                   scales: Optional[torch.Tensor] = None, residual_out: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None, plan: Optional[N.Plan] = None):
    """RMSNorm with MXFP8 output: returns (codes uint8 [rows, hidden] E4M3,
    scales uint8 [rows, hidden/32] E8M0) and, with a residual, residual_out."""
    _check_tensor(x, "x", x)
    code = dtype_code(x.dtype)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    if w is not None and tuple(w.shape) != (hidden,):
        raise ValueError(f"w must have shape ({hidden},)")
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(tuple(x.shape[:-1]) + (hidden // 32,), dtype=torch.uint8, device=x.device)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    for name, t in (("w", w), ("residual", residual), ("residual_out", residual_out)):
        _check_tensor(t, name, x)
    for name, t in (("codes", codes), ("scales", scales)):
        if not t.is_cuda or t.dtype != torch.uint8 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA uint8 tensor")
    with torch.cuda.device(x.device):
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        N.rmsnorm_fwd_mxfp8(_ptr(x), _ptr(residual), _ptr(w), _ptr(codes), _ptr(scales), _ptr(residual_out), rows,
                            hidden, float(eps), float(weight_bias), code, plan, s.cuda_stream)
    return (codes, scales, residual_out) if residual is not None else (codes, scales)


def rms_norm_mxfp8_plan_for(x, w=None, residual=None) -> N.Plan:
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    codes = torch.empty(1, dtype=torch.uint8, device=x.device)   # only its alignment matters
    with torch.cuda.device(x.device):
        return N.rmsnorm_mxfp8_plan_for(_ptr(x), _ptr(residual), _ptr(w), codes.data_ptr(), codes.data_ptr(),
                                        _ptr(residual), rows, hidden, dtype_code(x.dtype))


def rms_norm_nvfp4(x: torch.Tensor, w: Optional[torch.Tensor] = None, residual: Optional[torch.Tensor] = None,
                   eps: float = 1e-6, tensor_scale: float = 1.0, weight_bias: float = 0.0,
                   codes: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
                   residual_out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                   plan: Optional[N.Plan] = None):
    """RMSNorm with NVFP4 output (bf16 input): returns (codes uint8 [rows,
    hidden/2] with two E2M1 codes a byte, scales uint8 [rows, hidden/16]
    E4M3) and, with a residual, residual_out."""
    _check_tensor(x, "x", x)
    code = dtype_code(x.dtype)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    if w is not None and tuple(w.shape) != (hidden,):
        raise ValueError(f"w must have shape ({hidden},)")
    if codes is None:
        codes = torch.empty(tuple(x.shape[:-1]) + (hidden // 2,), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(tuple(x.shape[:-1]) + (hidden // 16,), dtype=torch.uint8, device=x.device)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    for name, t in (("w", w), ("residual", residual), ("residual_out", residual_out)):
        _check_tensor(t, name, x)
    for name, t in (("codes", codes), ("scales", scales)):
        if not t.is_cuda or t.dtype != torch.uint8 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA uint8 tensor")
    with torch.cuda.device(x.device):
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        N.rmsnorm_fwd_nvfp4(_ptr(x), _ptr(residual), _ptr(w), _ptr(codes), _ptr(scales), _ptr(residual_out), rows,
                            hidden, float(eps), float(weight_bias), float(tensor_scale), code, plan, s.cuda_stream)
    return (codes, scales, residual_out) if residual is not None else (codes, scales)


def rms_norm_nvfp4_plan_for(x, w=None, residual=None) -> N.Plan:
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    codes = torch.empty(1, dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        return N.rmsnorm_nvfp4_plan_for(_ptr(x), _ptr(residual), _ptr(w), codes.data_ptr(), codes.data_ptr(),
                                        _ptr(residual), rows, hidden, dtype_code(x.dtype))
