// kernel_table.h -- lookup of the compiled kernel instantiations (internal).
#pragma once

namespace rrn {

// Threads per row / chunk bounds compiled for the register kernel.
constexpr int kRegMaxGT = 512;
constexpr int kRegMaxCH = 8;
// Block sizes compiled for the two-pass kernel.
constexpr int kLoopBlocks[3] = {64, 256, 1024};

// dtype: 0 = f32, 1 = bf16.  Return the __global__ function as a launchable
// pointer, or nullptr when that combination is not compiled.
const void *reg_kernel_f32(int gt, int ch, bool res, bool w);
const void *reg_kernel_bf16(int gt, int ch, bool res, bool w);
const void *loop_kernel_f32(int block, bool vec, bool res, bool w);
const void *loop_kernel_bf16(int block, bool vec, bool res, bool w);

}  // namespace rrn
