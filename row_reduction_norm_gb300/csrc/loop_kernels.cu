// loop_kernels.cu -- instantiations of the two-pass kernel (both I/O types).
#include "kernel_table.h"
#include "rmsnorm_kernels.cuh"

namespace rrn {
namespace {

template <typename T, int VE, int BLOCK>
const void *pick(bool res, bool w) {
    if (res && w) return reinterpret_cast<const void *>(&rms_loop_kernel<T, VE, BLOCK, true, true>);
    if (res) return reinterpret_cast<const void *>(&rms_loop_kernel<T, VE, BLOCK, true, false>);
    if (w) return reinterpret_cast<const void *>(&rms_loop_kernel<T, VE, BLOCK, false, true>);
    return reinterpret_cast<const void *>(&rms_loop_kernel<T, VE, BLOCK, false, false>);
}

template <typename T>
const void *pick_block(int block, bool vec, bool res, bool w) {
    switch (block) {
        case 64: return vec ? pick<T, T::kVec, 64>(res, w) : pick<T, 1, 64>(res, w);
        case 256: return vec ? pick<T, T::kVec, 256>(res, w) : pick<T, 1, 256>(res, w);
        case 1024: return vec ? pick<T, T::kVec, 1024>(res, w) : pick<T, 1, 1024>(res, w);
        default: return nullptr;
    }
}

}  // namespace

const void *loop_kernel_f32(int block, bool vec, bool res, bool w) {
    return pick_block<F32>(block, vec, res, w);
}
const void *loop_kernel_bf16(int block, bool vec, bool res, bool w) {
    return pick_block<BF16>(block, vec, res, w);
}

}  // namespace rrn
