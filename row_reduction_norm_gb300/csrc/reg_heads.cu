// reg_heads.cu -- register-kernel instantiations for head rows (fused Q+K norm).
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *reg_heads_f32(int gt, int ch, int wm) { return pick::reg_gt<F32, false, true, kRegMaxGTHeads>(gt, ch, wm); }
const void *reg_heads_bf16(int gt, int ch, int wm) { return pick::reg_gt<BF16, false, true, kRegMaxGTHeads>(gt, ch, wm); }

}  // namespace rrn
