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
             plan: Optional[N.Plan] = None):
    """y = x * rsqrt(mean(x^2) + eps) * w over the last dimension.

    With ``residual``: h = x + residual (rounded to the I/O type) is written to
    ``residual_out`` and normalised; returns ``(y, residual_out)``.  Without:
    returns ``y``.  ``plan`` forces a launch plan (see ``rmsnorm_fwd_plan``).
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
                float(eps), code)
        if plan is None:
            N.rmsnorm_fwd(*args, s.cuda_stream)
        else:
            N.rmsnorm_fwd_plan(*args, plan, s.cuda_stream)
    return (y, residual_out) if residual is not None else y


def plan_for(x: torch.Tensor, w=None, residual=None, out=None, residual_out=None) -> N.Plan:
    """The plan ``rms_norm`` would launch for these tensors."""
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    y = out if out is not None else x
    ro = residual_out if residual_out is not None else residual
    with torch.cuda.device(x.device):
        return N.rmsnorm_plan_for(_ptr(x), _ptr(residual), _ptr(w), _ptr(y), _ptr(ro), rows, hidden,
                                  dtype_code(x.dtype))
