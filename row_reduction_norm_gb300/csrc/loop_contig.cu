// loop_contig.cu -- two-pass kernel instantiations for contiguous rows.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *loop_contig(int dtype, int block, bool vec, bool res, int wm) {
    if (dtype == 1)
        return res ? pick::loop_block<BF16, true, false>(block, vec, wm) : pick::loop_block<BF16, false, false>(block, vec, wm);
    return res ? pick::loop_block<F32, true, false>(block, vec, wm) : pick::loop_block<F32, false, false>(block, vec, wm);
}

}  // namespace rrn
