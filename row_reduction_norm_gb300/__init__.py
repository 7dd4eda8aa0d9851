"""row_reduction_norm_gb300 -- fused row-wise RMSNorm (and LayerNorm) for GB300 (sm_103a).

``y = x * rsqrt(mean(x^2) + eps) * w`` per row, with an optional fused
residual add and an optional weight, bf16 or fp32 I/O.  The work runs in
hand-written CUDA kernels behind the C ABI of ``include/rmsnorm.h``
(``librmsnorm_gb300.so``, built with ``python -m row_reduction_norm_gb300.build``);
this package is the thin binding over it.  Importing it loads nothing: the
library is loaded at the first call, and a missing library is an error.
"""
from ._native import (  # noqa: F401  (the C ABI, same names)
    Plan, RmsNormError, rmsnorm_build_info, rmsnorm_fwd, rmsnorm_fwd_ex, rmsnorm_fwd_plan, rmsnorm_fwd_cast,
    rmsnorm_max_hidden, rmsnorm_plan, rmsnorm_plan_ex, rmsnorm_plan_for, rmsnorm_regime, rmsnorm_qk_fwd, rmsnorm_qk_plan_for,
    layernorm_fwd, layernorm_plan_for, rmsnorm_fwd_mxfp8, rmsnorm_mxfp8_plan_for, rmsnorm_fwd_nvfp4,
    rmsnorm_nvfp4_plan_for, rmsnorm_fwd_host, rmsnorm_host_workspace_bytes, rmsnorm_fwd_host_static,
    rmsnorm_reg_max_chunks, rmsnorm_wait_timeouts, rmsnorm_strerror,
    RMSNORM_BF16, RMSNORM_F32, RMSNORM_OK, RMSNORM_EINVAL, RMSNORM_EUNSUPPORTED, RMSNORM_ECUDA,
)
from .api import (  # noqa: F401
    rms_norm, plan_for, qk_norm, qk_plan_for, layer_norm, layer_norm_plan_for, rms_norm_mxfp8,
    rms_norm_mxfp8_plan_for, rms_norm_nvfp4, rms_norm_nvfp4_plan_for, rms_norm_host, dtype_code)

__version__ = "0.1.0"
