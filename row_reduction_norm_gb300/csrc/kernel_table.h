// kernel_table.h -- lookup of the compiled kernel instantiations (internal).
#pragma once

namespace rrn {

// Threads per row / chunk bounds compiled for the register kernel.
constexpr int kRegMaxGT = 512;        // contiguous rows
constexpr int kRegMaxGTHeads = 32;    // head rows (heads are short)
constexpr int kRegMaxCH = 8;
// Block sizes compiled for the two-pass kernel.
constexpr int kLoopBlocks[3] = {64, 256, 1024};

// dtype: 0 = f32, 1 = bf16; wm: 0 no weight, 1 weight, 2 weight + bias.
// Each returns the __global__ function as a launchable pointer, or nullptr
// when that combination is not compiled.
const void *reg_contig_f32_plain(int gt, int ch, int wm);
const void *reg_contig_f32_res(int gt, int ch, int wm);
const void *reg_contig_bf16_plain(int gt, int ch, int wm);
const void *reg_contig_bf16_res(int gt, int ch, int wm);
const void *reg_heads_f32(int gt, int ch, int wm);
const void *reg_heads_bf16(int gt, int ch, int wm);
const void *loop_contig(int dtype, int block, bool vec, bool res, int wm);
const void *loop_heads(int dtype, int block, bool vec, int wm);

// RMSNorm with MXFP8 output (contiguous rows, register kernel only).
const void *mx_reg_f32_plain(int gt, int ch, int wm);
const void *mx_reg_f32_res(int gt, int ch, int wm);
const void *mx_reg_bf16_plain(int gt, int ch, int wm);
const void *mx_reg_bf16_res(int gt, int ch, int wm);

inline const void *mx_kernel(int dtype, int gt, int ch, bool res, int wm) {
    if (dtype == 1) return res ? mx_reg_bf16_res(gt, ch, wm) : mx_reg_bf16_plain(gt, ch, wm);
    return res ? mx_reg_f32_res(gt, ch, wm) : mx_reg_f32_plain(gt, ch, wm);
}

// RMSNorm with NVFP4 output (bf16 I/O, contiguous rows, register kernel only).
const void *nv_reg_bf16_plain(int gt, int ch, int wm);
const void *nv_reg_bf16_res(int gt, int ch, int wm);

inline const void *nv_kernel(int dtype, int gt, int ch, bool res, int wm) {
    if (dtype != 1) return nullptr;
    return res ? nv_reg_bf16_res(gt, ch, wm) : nv_reg_bf16_plain(gt, ch, wm);
}

// LayerNorm (contiguous rows); aff: 0 none, 1 weight, 2 weight and bias.
constexpr int kLnMaxGT = 256;
const void *ln_reg_f32(int gt, int ch, bool res, int aff);
const void *ln_reg_bf16(int gt, int ch, bool res, int aff);
const void *ln_loop(int dtype, int block, bool vec, bool res, int aff);

inline const void *reg_kernel(int dtype, int gt, int ch, bool res, int wm, bool heads) {
    if (heads) return res ? nullptr : (dtype == 1 ? reg_heads_bf16(gt, ch, wm) : reg_heads_f32(gt, ch, wm));
    if (dtype == 1) return res ? reg_contig_bf16_res(gt, ch, wm) : reg_contig_bf16_plain(gt, ch, wm);
    return res ? reg_contig_f32_res(gt, ch, wm) : reg_contig_f32_plain(gt, ch, wm);
}

inline const void *loop_kernel(int dtype, int block, bool vec, bool res, int wm, bool heads) {
    if (heads) return res ? nullptr : loop_heads(dtype, block, vec, wm);
    return loop_contig(dtype, block, vec, res, wm);
}

}  // namespace rrn
