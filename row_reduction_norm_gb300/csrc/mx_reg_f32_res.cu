// mx_reg_f32_res.cu -- RMSNorm with MXFP8 output: register-kernel instantiations, f32 I/O, fused residual add.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *mx_reg_f32_res(int gt, int ch, int wm) { return pick::mx_gt<F32, true>(gt, ch, wm); }

}  // namespace rrn
