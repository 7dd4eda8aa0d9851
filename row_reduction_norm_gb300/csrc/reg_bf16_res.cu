// reg_bf16_res.cu -- register-kernel instantiations: bf16 I/O, contiguous rows, fused residual add.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *reg_contig_bf16_res(int gt, int ch, int wm) {
    return pick::reg_gt<BF16, true, false, kRegMaxGT>(gt, ch, wm);
}

}  // namespace rrn
