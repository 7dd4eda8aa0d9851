// ln_reg_bf16.cu -- LayerNorm register-kernel instantiations, bf16 I/O.
#include "kernel_table.h"
#include "ln_pick.cuh"

namespace rrn {

const void *ln_reg_bf16(int gt, int ch, bool res, int aff) {
    return res ? lnpick::reg_gt<BF16, true>(gt, ch, aff) : lnpick::reg_gt<BF16, false>(gt, ch, aff);
}

}  // namespace rrn
