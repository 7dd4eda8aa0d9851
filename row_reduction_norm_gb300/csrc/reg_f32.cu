// reg_f32.cu -- instantiations of the register kernel for the f32 I/O type.
#include "kernel_table.h"
#include "rmsnorm_kernels.cuh"

namespace rrn {
namespace {

template <int GT, int CH>
const void *pick(bool res, bool w) {
    if (res && w) return reinterpret_cast<const void *>(&rms_reg_kernel<F32, GT, CH, true, true>);
    if (res) return reinterpret_cast<const void *>(&rms_reg_kernel<F32, GT, CH, true, false>);
    if (w) return reinterpret_cast<const void *>(&rms_reg_kernel<F32, GT, CH, false, true>);
    return reinterpret_cast<const void *>(&rms_reg_kernel<F32, GT, CH, false, false>);
}

template <int GT>
const void *pick_ch(int ch, bool res, bool w) {
    switch (ch) {
        case 1: return pick<GT, 1>(res, w);
        case 2: return pick<GT, 2>(res, w);
        case 4: return pick<GT, 4>(res, w);
        case 8: return pick<GT, 8>(res, w);
        default: return nullptr;
    }
}

}  // namespace

const void *reg_kernel_f32(int gt, int ch, bool res, bool w) {
    switch (gt) {
        case 4: return pick_ch<4>(ch, res, w);
        case 8: return pick_ch<8>(ch, res, w);
        case 16: return pick_ch<16>(ch, res, w);
        case 32: return pick_ch<32>(ch, res, w);
        case 64: return pick_ch<64>(ch, res, w);
        case 128: return pick_ch<128>(ch, res, w);
        case 256: return pick_ch<256>(ch, res, w);
        case 512: return pick_ch<512>(ch, res, w);
        default: return nullptr;
    }
}

}  // namespace rrn
