// ln_reg_f32.cu -- LayerNorm register-kernel instantiations, f32 I/O.
#include "kernel_table.h"
#include "ln_pick.cuh"

namespace rrn {

const void *ln_reg_f32(int gt, int ch, bool res, int aff) {
    return res ? lnpick::reg_gt<F32, true>(gt, ch, aff) : lnpick::reg_gt<F32, false>(gt, ch, aff);
}

}  // namespace rrn
