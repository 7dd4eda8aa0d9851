// cast_bf16.cu -- register- and two-pass-kernel instantiations of the
// cast-order weight mode: bf16 I/O, contiguous rows, with and without a residual.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *reg_contig_bf16_cast(int gt, int ch, bool res) {
    return res ? pick::reg_gt<BF16, true, false, kRegMaxGT, true>(gt, ch, kWeightCast)
               : pick::reg_gt<BF16, false, false, kRegMaxGT, true>(gt, ch, kWeightCast);
}

const void *loop_contig_bf16_cast(int block, bool vec, bool res) {
    return res ? pick::loop_block<BF16, true, false, true>(block, vec, kWeightCast)
               : pick::loop_block<BF16, false, false, true>(block, vec, kWeightCast);
}

}  // namespace rrn
