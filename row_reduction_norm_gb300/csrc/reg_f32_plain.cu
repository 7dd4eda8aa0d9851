// reg_f32_plain.cu -- register-kernel instantiations: f32 I/O, contiguous rows, no residual.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *reg_contig_f32_plain(int gt, int ch, int wm) {
    return pick::reg_gt<F32, false, false, kRegMaxGT>(gt, ch, wm);
}

}  // namespace rrn
