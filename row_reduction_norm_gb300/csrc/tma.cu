// tma.cu -- instantiations of the shared-memory (bulk copy) RMSNorm kernel,
// and the device counter its bounded waits report to.
#include <type_traits>

#include "kernel_table.h"
#include "rmsnorm_tma.cuh"

namespace rrn {
namespace {

template <typename T, bool RES, int PC, int OUT>
const void *tma_wm(int wm) {
    switch (wm) {
        case kNoWeight: return reinterpret_cast<const void *>(&rms_tma_kernel<T, RES, kNoWeight, PC, OUT>);
        case kWeight: return reinterpret_cast<const void *>(&rms_tma_kernel<T, RES, kWeight, PC, OUT>);
        case kWeightBias: return reinterpret_cast<const void *>(&rms_tma_kernel<T, RES, kWeightBias, PC, OUT>);
        case kWeightCast:
            if constexpr (std::is_same<T, BF16>::value && OUT == kOutT)
                return reinterpret_cast<const void *>(&rms_tma_kernel<T, RES, kWeightCast, PC, OUT>);
            else
                return nullptr;
        default: return nullptr;
    }
}

template <typename T, bool RES>
const void *tma_pc(int pc, int wm) {
    switch (pc) {
        case 1: return tma_wm<T, RES, 1, kOutT>(wm);
        case 2: return tma_wm<T, RES, 2, kOutT>(wm);
        case 4: return tma_wm<T, RES, 4, kOutT>(wm);
        default: return nullptr;
    }
}

}  // namespace

const void *tma_kernel(int dtype, int pc, bool res, int wm) {
    if (dtype == 1) return res ? tma_pc<BF16, true>(pc, wm) : tma_pc<BF16, false>(pc, wm);
    return res ? tma_pc<F32, true>(pc, wm) : tma_pc<F32, false>(pc, wm);
}

const void *tma_quant_kernel(int dtype, bool res, int wm, int out) {
    if (out == kOutMxfp8) {
        if (dtype == 1) return res ? tma_wm<BF16, true, 2, kOutMxfp8>(wm) : tma_wm<BF16, false, 2, kOutMxfp8>(wm);
        return res ? tma_wm<F32, true, 2, kOutMxfp8>(wm) : tma_wm<F32, false, 2, kOutMxfp8>(wm);
    }
    if (out == kOutNvfp4 && dtype == 1)
        return res ? tma_wm<BF16, true, 2, kOutNvfp4>(wm) : tma_wm<BF16, false, 2, kOutNvfp4>(wm);
    return nullptr;
}

int tma_timeouts_read(unsigned int *out) {
    return cudaMemcpyFromSymbol(out, g_tma_timeouts, sizeof(unsigned int)) == cudaSuccess ? 0 : -1;
}

}  // namespace rrn
