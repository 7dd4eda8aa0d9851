// mx_reg_f32_plain.cu -- RMSNorm with MXFP8 output: register-kernel instantiations, f32 I/O, no residual.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *mx_reg_f32_plain(int gt, int ch, int wm) { return pick::mx_gt<F32, false>(gt, ch, wm); }

}  // namespace rrn
