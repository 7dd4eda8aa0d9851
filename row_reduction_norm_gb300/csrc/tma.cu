// tma.cu -- instantiations of the shared-memory (bulk copy) RMSNorm kernel,
// and the device counter its bounded waits report to.
#include <type_traits>

#include "kernel_table.h"
#include "rmsnorm_tma.cuh"

namespace rrn {
namespace {

template <typename T, bool RES, int WM, int PC, int OUT>
const void *tma_wg(bool wg) {
    if constexpr (WM == kNoWeight)
        return reinterpret_cast<const void *>(&rms_tma_kernel<T, RES, WM, PC, OUT, false>);
    else
        return wg ? reinterpret_cast<const void *>(&rms_tma_kernel<T, RES, WM, PC, OUT, true>)
                  : reinterpret_cast<const void *>(&rms_tma_kernel<T, RES, WM, PC, OUT, false>);
}

template <typename T, bool RES, int PC, int OUT>
const void *tma_wm(int wm, bool wg) {
    switch (wm) {
        case kNoWeight: return tma_wg<T, RES, kNoWeight, PC, OUT>(wg);
        case kWeight: return tma_wg<T, RES, kWeight, PC, OUT>(wg);
        case kWeightBias: return tma_wg<T, RES, kWeightBias, PC, OUT>(wg);
        case kWeightCast:
            if constexpr (std::is_same<T, BF16>::value && OUT == kOutT)
                return tma_wg<T, RES, kWeightCast, PC, OUT>(wg);
            else
                return nullptr;
        default: return nullptr;
    }
}

template <typename T, bool RES>
const void *tma_pc(int pc, int wm, bool wg) {
    switch (pc) {
        case 1: return tma_wm<T, RES, 1, kOutT>(wm, wg);
        case 2: return tma_wm<T, RES, 2, kOutT>(wm, wg);
        case 4: return tma_wm<T, RES, 4, kOutT>(wm, wg);
        default: return nullptr;
    }
}

}  // namespace

const void *tma_kernel(int dtype, int pc, bool res, int wm, bool wg) {
    if (dtype == 1) return res ? tma_pc<BF16, true>(pc, wm, wg) : tma_pc<BF16, false>(pc, wm, wg);
    return res ? tma_pc<F32, true>(pc, wm, wg) : tma_pc<F32, false>(pc, wm, wg);
}

const void *tma_quant_kernel(int dtype, bool res, int wm, int out, bool wg) {
    if (out == kOutMxfp8) {
        if (dtype == 1)
            return res ? tma_wm<BF16, true, 2, kOutMxfp8>(wm, wg) : tma_wm<BF16, false, 2, kOutMxfp8>(wm, wg);
        return res ? tma_wm<F32, true, 2, kOutMxfp8>(wm, wg) : tma_wm<F32, false, 2, kOutMxfp8>(wm, wg);
    }
    if (out == kOutNvfp4 && dtype == 1)
        return res ? tma_wm<BF16, true, 2, kOutNvfp4>(wm, wg) : tma_wm<BF16, false, 2, kOutNvfp4>(wm, wg);
    return nullptr;
}

int tma_timeouts_read(unsigned int *out) {
    return cudaMemcpyFromSymbol(out, g_tma_timeouts, sizeof(unsigned int)) == cudaSuccess ? 0 : -1;
}

}  // namespace rrn
