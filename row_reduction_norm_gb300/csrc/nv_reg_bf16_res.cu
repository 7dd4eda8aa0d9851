// nv_reg_bf16_res.cu -- RMSNorm with NVFP4 output: register-kernel instantiations, bf16 I/O, fused residual add.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *nv_reg_bf16_res(int gt, int ch, int wm) { return pick::nv_gt<BF16, true>(gt, ch, wm); }

}  // namespace rrn
