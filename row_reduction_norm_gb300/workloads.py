"""Seeded synthetic inputs for the fused RMSNorm, shared by the tests and the benchmark.

This module holds no arithmetic of the method: it only draws random tensors
and rounds them once to the I/O type.  Both the CUDA path and the CPU oracle
receive the identical bits from here.

The shapes stand in for the models the pages run: width 576 (SmolLM2-135M) and
2048 (Llama-3.2-1B) from the model-as-a-kernel card ("Measured"), and the
per-head qk-norm over 128-element heads (Qwen3 style) from "CuTeDSL at
Perplexity", section "QK Norm".  Distributions are written N(mean, std).

Recipe: each tensor is drawn in fp32 from its own ``torch.Generator`` on the
requested device, seeded ``seed`` (x), ``seed+1`` (residual), ``seed+2`` (w) and
``seed+3`` (outlier mask), scaled and shifted as listed, then rounded once to
the I/O type.  Outliers: an independent Bernoulli(p) mask multiplies the
selected entries of x by ``outlier_scale`` before the rounding.  The random
stream differs between CPU and CUDA generators, so a given (seed, device)
pair names one input set; parity checks always hand the same tensors to both
sides.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "bf16" | "f32" (I/O type of every tensor)
    rows: int
    hidden: int
    eps: float
    x_std: float
    res_std: Optional[float]   # None: no fused residual add
    w_std: Optional[float]     # None: no weight (w ~ 1 + N(0, w_std) otherwise)
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    note: str = ""
    b_std: Optional[float] = None   # LayerNorm bias ~ N(0, b_std) (None: no bias)
    x_mean: float = 0.0             # x ~ x_mean + N(0, x_std)

    @property
    def has_res(self) -> bool:
        return self.res_std is not None

    @property
    def has_w(self) -> bool:
        return self.w_std is not None

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def has_b(self) -> bool:
        return self.b_std is not None

    def algorithmic_bytes(self, rows: Optional[int] = None) -> int:
        """Bytes one pass must move: read x (+ residual), write y (+ residual_out), read w (and b) once."""
        r = self.rows if rows is None else rows
        per_row = self.hidden * self.elem_bytes * (2 + (2 if self.has_res else 0))
        return r * per_row + self.hidden * self.elem_bytes * ((1 if self.has_w else 0) + (1 if self.has_b else 0))

    def with_rows(self, rows: int) -> "Workload":
        return dataclasses.replace(self, rows=rows, name=f"{self.name}@rows={rows}")


WORKLOADS = {
    w.name: w
    for w in [
        Workload("f32_64x256", "f32", 64, 256, 1e-6, 1.0, None, 0.1,
                 note="small case the oracle finishes at once"),
        Workload("bf16_4096x576", "bf16", 4096, 576, 1e-5, 1.0, None, 0.05,
                 note="SmolLM2-135M width, warp-per-row"),
        Workload("bf16_res_16384x2048", "bf16", 16384, 2048, 1e-5, 0.5, 1.0, 0.05,
                 note="Llama-3.2-1B width, fused residual add"),
        Workload("bf16_qk_262144x128", "bf16", 262144, 128, 1e-6, 2.0, None, 0.1,
                 note="per-head qk-norm, 8192 tokens x 32 heads, shared weight"),
        Workload("bf16_decode_1x4096", "bf16", 1, 4096, 1e-6, 2.0, None, 0.1, note="decode latency"),
        Workload("bf16_decode_8x4096", "bf16", 8, 4096, 1e-6, 2.0, None, 0.1, note="decode latency"),
        Workload("bf16_decode_64x4096", "bf16", 64, 4096, 1e-6, 2.0, None, 0.1, note="decode latency"),
        Workload("bf16_res_65536x8192_w", "bf16", 65536, 8192, 1e-6, 1.0, 1.0, 0.1,
                 outlier_frac=1e-3, outlier_scale=100.0,
                 note="bandwidth-roofline case with outliers, weight"),
        Workload("bf16_res_65536x8192_nw", "bf16", 65536, 8192, 1e-6, 1.0, 1.0, None,
                 outlier_frac=1e-3, outlier_scale=100.0,
                 note="bandwidth-roofline case with outliers, no weight"),
        # rows too long for registers (not among the pages' model widths):
        # the shared-memory (bulk copy) regime and the two-pass regime
        Workload("bf16_4096x32768_w", "bf16", 4096, 32768, 1e-6, 1.0, None, 0.1,
                 note="long rows, shared-memory regime, weight resident"),
        Workload("bf16_res_4096x40960_w", "bf16", 4096, 40960, 1e-6, 1.0, 1.0, 0.1,
                 note="longest rows of the shared-memory regime (80 KB), fused residual"),
        Workload("bf16_2048x65536_w", "bf16", 2048, 65536, 1e-6, 1.0, None, 0.1,
                 note="longest bf16 rows without a residual, shared-memory regime, weight streamed"),
        Workload("bf16_res_2048x65536_w", "bf16", 2048, 65536, 1e-6, 1.0, 1.0, 0.1,
                 note="longest bf16 rows, two-pass regime"),
        Workload("f32_res_2048x65536_w", "f32", 2048, 65536, 1e-6, 1.0, 1.0, 0.1,
                 note="longest fp32 rows, two-pass regime"),
    ]
}

TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_inputs(wl: Workload, seed: int = 0, device="cpu", rows: Optional[int] = None):
    """Draw (x, residual, w) for ``wl`` as tensors of the I/O type on ``device``.

    ``residual`` and ``w`` are None when the workload has none.  ``rows``
    overrides the row count (same distributions).
    """
    device = torch.device(device)
    r = wl.rows if rows is None else int(rows)
    h = wl.hidden
    dt = TORCH_DTYPE[wl.dtype]
    x = torch.randn((r, h), generator=_gen(device, seed), device=device, dtype=torch.float32)
    x.mul_(wl.x_std)
    if wl.x_mean:
        x.add_(wl.x_mean)
    if wl.outlier_frac > 0.0:
        u = torch.rand((r, h), generator=_gen(device, seed + 3), device=device, dtype=torch.float32)
        x = torch.where(u < wl.outlier_frac, x * wl.outlier_scale, x)
        del u
    x = x.to(dt)
    residual = None
    if wl.has_res:
        residual = torch.randn((r, h), generator=_gen(device, seed + 1), device=device,
                               dtype=torch.float32).mul_(wl.res_std).to(dt)
    w = None
    if wl.has_w:
        w = (torch.randn((h,), generator=_gen(device, seed + 2), device=device,
                         dtype=torch.float32).mul_(wl.w_std).add_(1.0)).to(dt)
    return x, residual, w


def random_rows(dtype: str, rows: int, hidden: int, seed: int, device="cpu", std: float = 1.0):
    """Plain N(0, std) rows in the I/O type (edge-case and sweep tests)."""
    t = torch.randn((rows, hidden), generator=_gen(torch.device(device), seed),
                    device=device, dtype=torch.float32).mul_(std)
    return t.to(TORCH_DTYPE[dtype])


def to_numpy_bits(t: Optional[torch.Tensor]):
    """Host numpy view of a tensor in the oracle's convention (bf16 -> uint16 bits)."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def from_numpy_bits(a, dtype: str) -> torch.Tensor:
    """Inverse of ``to_numpy_bits`` (CPU tensor)."""
    if dtype == "bf16":
        return torch.from_numpy(a.view("int16").copy()).view(torch.bfloat16)
    return torch.from_numpy(a.copy())


@dataclasses.dataclass(frozen=True)
class QKWorkload:
    """Packed token rows [q heads | k heads | v heads] for the fused Q+K norm."""
    name: str
    dtype: str
    tokens: int
    q_heads: int
    k_heads: int
    v_heads: int
    head_dim: int
    eps: float
    x_std: float
    w_std: Optional[float]        # None: no weights
    weight_bias: float = 0.0      # added to every weight element
    w_mean: float = 1.0           # weights ~ w_mean + N(0, w_std)
    note: str = ""

    @property
    def width(self) -> int:
        return (self.q_heads + self.k_heads + self.v_heads) * self.head_dim

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def algorithmic_bytes(self) -> int:
        """Read and write every query and key head once, read both weights."""
        heads = self.tokens * (self.q_heads + self.k_heads)
        w = 2 * self.head_dim * self.elem_bytes if self.w_std is not None else 0
        return heads * self.head_dim * self.elem_bytes * 2 + w


QK_WORKLOADS = {
    w.name: w
    for w in [
        QKWorkload("qk_bf16_8192tok_q32_k8_v8_hd128", "bf16", 8192, 32, 8, 8, 128, 1e-6, 2.0, 0.1,
                   note="Qwen3-8B-like fused projection, query and key norms in one launch"),
        QKWorkload("qk_bf16_8192tok_q32_k8_v8_hd128_1pw", "bf16", 8192, 32, 8, 8, 128, 1e-6, 2.0, 0.1,
                   weight_bias=1.0, w_mean=0.0, note="same, (1 + w) weight form"),
        QKWorkload("qk_bf16_64tok_q32_k8_v8_hd128", "bf16", 64, 32, 8, 8, 128, 1e-6, 2.0, 0.1,
                   note="decode batch"),
    ]
}


def make_qk_inputs(wl: QKWorkload, seed: int = 0, device="cpu", tokens: Optional[int] = None,
                   stride: Optional[int] = None):
    """Draw (qkv, q_w, k_w): qkv [tokens, stride] (stride >= width; value heads and
    padding drawn like the rest), weights ~ w_mean + N(0, w_std) or None."""
    device = torch.device(device)
    t = wl.tokens if tokens is None else int(tokens)
    width = wl.width if stride is None else int(stride)
    dt = TORCH_DTYPE[wl.dtype]
    qkv = torch.randn((t, width), generator=_gen(device, seed), device=device,
                      dtype=torch.float32).mul_(wl.x_std).to(dt)
    q_w = k_w = None
    if wl.w_std is not None:
        q_w = (torch.randn((wl.head_dim,), generator=_gen(device, seed + 2), device=device,
                           dtype=torch.float32).mul_(wl.w_std).add_(wl.w_mean)).to(dt)
        k_w = (torch.randn((wl.head_dim,), generator=_gen(device, seed + 4), device=device,
                           dtype=torch.float32).mul_(wl.w_std).add_(wl.w_mean)).to(dt)
    return qkv, q_w, k_w


# LayerNorm workloads: GPT-2 (width 768, eps 1e-5, weight and bias) from "GPT-2
# on the GPU", section "The Whole Model as One Kernel", plus a wider fused
# residual case.  Weights ~ 1 + N(0, 0.1), biases ~ N(0, 0.1).
LN_WORKLOADS = {
    w.name: w
    for w in [
        Workload("ln_f32_64x768_wb", "f32", 64, 768, 1e-5, 1.0, None, 0.1, b_std=0.1,
                 note="GPT-2 width, fp32 as the tutorial runs it"),
        Workload("ln_bf16_16384x768_wb", "bf16", 16384, 768, 1e-5, 1.0, None, 0.1, b_std=0.1, x_mean=0.5,
                 note="GPT-2 width, 16384 tokens"),
        Workload("ln_bf16_res_16384x4096_wb", "bf16", 16384, 4096, 1e-5, 1.0, 1.0, 0.1, b_std=0.1,
                 note="fused residual add, width 4096"),
    ]
}


def make_ln_inputs(wl: Workload, seed: int = 0, device="cpu", rows: Optional[int] = None):
    """(x, residual, w, b) for a LayerNorm workload; b drawn with seed + 5."""
    x, r, w = make_inputs(wl, seed=seed, device=device, rows=rows)
    b = None
    if wl.has_b:
        dev = torch.device(device)
        b = torch.randn((wl.hidden,), generator=_gen(dev, seed + 5), device=dev,
                        dtype=torch.float32).mul_(wl.b_std).to(TORCH_DTYPE[wl.dtype])
    return x, r, w, b


# RMSNorm in the op-by-op cast order (normalised value rounded to bf16 before
# the weight multiply): the same data as three plain-order rows, one per
# kernel family the library plans for them (CTA registers, CTA registers at
# the bandwidth case, shared-memory rings).
CAST_WORKLOADS = {
    "cast_" + name: dataclasses.replace(WORKLOADS[name], name="cast_" + name,
                                        note=WORKLOADS[name].note + ", cast order")
    for name in ("bf16_res_16384x2048", "bf16_res_65536x8192_w", "bf16_res_4096x40960_w")
}


# RMSNorm with MXFP8 output (E4M3 codes + one E8M0 scale per 32 elements):
# the Llama-3.2-1B-width residual case and the 65536 x 8192 bandwidth case.
MX_WORKLOADS = {
    w.name: w
    for w in [
        Workload("mx_bf16_res_16384x2048", "bf16", 16384, 2048, 1e-5, 0.5, 1.0, 0.05,
                 note="fused residual add, MXFP8 output"),
        Workload("mx_bf16_res_65536x8192_w", "bf16", 65536, 8192, 1e-6, 1.0, 1.0, 0.1,
                 outlier_frac=1e-3, outlier_scale=100.0, note="bandwidth case, MXFP8 output"),
    ]
}


def mx_algorithmic_bytes(wl: Workload) -> int:
    """Read x (+ residual), write the codes (1 byte an element) and scales (1 per
    32) (+ residual_out), read w once."""
    e = wl.rows * wl.hidden
    b = e * wl.elem_bytes * (1 + (2 if wl.has_res else 0)) + e + e // 32
    return b + (wl.hidden * wl.elem_bytes if wl.has_w else 0)


# RMSNorm with NVFP4 output (bf16 in): the same shapes as the MXFP8 rows, with a
# per-tensor scale of 1/64 (block scales stay inside E4M3's range for these
# distributions: amax / (6 S) <= 448 for amax up to 42).
NV_TENSOR_SCALE = 1.0 / 64.0
NV_WORKLOADS = {
    w.name: w
    for w in [
        Workload("nv_bf16_res_16384x2048", "bf16", 16384, 2048, 1e-5, 0.5, 1.0, 0.05,
                 note="fused residual add, NVFP4 output"),
        Workload("nv_bf16_res_65536x8192_w", "bf16", 65536, 8192, 1e-6, 1.0, 1.0, 0.1,
                 outlier_frac=1e-3, outlier_scale=100.0, note="bandwidth case, NVFP4 output"),
    ]
}


def nv_algorithmic_bytes(wl: Workload) -> int:
    """Read x (+ residual), write the codes (half a byte an element) and scales
    (1 per 16) (+ residual_out), read w once."""
    e = wl.rows * wl.hidden
    b = e * wl.elem_bytes * (1 + (2 if wl.has_res else 0)) + e // 2 + e // 16
    return b + (wl.hidden * wl.elem_bytes if wl.has_w else 0)
