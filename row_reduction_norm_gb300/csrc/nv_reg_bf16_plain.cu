// nv_reg_bf16_plain.cu -- RMSNorm with NVFP4 output: register-kernel instantiations, bf16 I/O, no residual.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *nv_reg_bf16_plain(int gt, int ch, int wm) { return pick::nv_gt<BF16, false>(gt, ch, wm); }

}  // namespace rrn
