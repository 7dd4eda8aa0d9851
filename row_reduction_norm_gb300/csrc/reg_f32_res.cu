// reg_f32_res.cu -- register-kernel instantiations: f32 I/O, contiguous rows, fused residual add.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *reg_contig_f32_res(int gt, int ch, int wm) {
    return pick::reg_gt<F32, true, false, kRegMaxGT>(gt, ch, wm);
}

}  // namespace rrn
