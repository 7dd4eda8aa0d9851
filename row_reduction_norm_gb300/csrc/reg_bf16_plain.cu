// reg_bf16_plain.cu -- register-kernel instantiations: bf16 I/O, contiguous rows, no residual.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *reg_contig_bf16_plain(int gt, int ch, int wm) {
    return pick::reg_gt<BF16, false, false, kRegMaxGT>(gt, ch, wm);
}

}  // namespace rrn
