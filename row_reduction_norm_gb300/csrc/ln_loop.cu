// ln_loop.cu -- LayerNorm three-pass kernel instantiations (both I/O types).
#include "kernel_table.h"
#include "ln_pick.cuh"

namespace rrn {

const void *ln_loop(int dtype, int block, bool vec, bool res, int aff) {
    if (dtype == 1)
        return res ? lnpick::loop_block<BF16, true>(block, vec, aff) : lnpick::loop_block<BF16, false>(block, vec, aff);
    return res ? lnpick::loop_block<F32, true>(block, vec, aff) : lnpick::loop_block<F32, false>(block, vec, aff);
}

}  // namespace rrn
