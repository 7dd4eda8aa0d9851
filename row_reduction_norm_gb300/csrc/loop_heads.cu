// loop_heads.cu -- two-pass kernel instantiations for head rows.
#include "kernel_pick.cuh"
#include "kernel_table.h"

namespace rrn {

const void *loop_heads(int dtype, int block, bool vec, int wm) {
    return dtype == 1 ? pick::loop_block<BF16, false, true>(block, vec, wm) : pick::loop_block<F32, false, true>(block, vec, wm);
}

}  // namespace rrn
