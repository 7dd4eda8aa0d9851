// cluster.cu -- instantiations of the cluster kernel (contiguous rows with a
// residual, a row split over the blocks of a thread-block cluster).
#include <type_traits>

#include "kernel_table.h"
#include "rmsnorm_cluster.cuh"

namespace rrn {
namespace {

template <typename T, int CH>
const void *cluster_wm(int wm) {
    switch (wm) {
        case kNoWeight: return reinterpret_cast<const void *>(&rms_cluster_kernel<T, CH, true, kNoWeight>);
        case kWeight: return reinterpret_cast<const void *>(&rms_cluster_kernel<T, CH, true, kWeight>);
        case kWeightBias: return reinterpret_cast<const void *>(&rms_cluster_kernel<T, CH, true, kWeightBias>);
        case kWeightCast:
            if constexpr (std::is_same<T, BF16>::value)
                return reinterpret_cast<const void *>(&rms_cluster_kernel<T, CH, true, kWeightCast>);
            else
                return nullptr;
        default: return nullptr;
    }
}

}  // namespace

const void *cluster_kernel(int dtype, int ch, bool res, int wm) {
    if (!res) return nullptr;
    if (dtype == 1) {
        if (ch == 4) return cluster_wm<BF16, 4>(wm);
        if (ch == 5) return cluster_wm<BF16, 5>(wm);
        return nullptr;
    }
    if (ch == 4) return cluster_wm<F32, 4>(wm);
    if (ch == 5) return cluster_wm<F32, 5>(wm);
    if (ch == 8) return cluster_wm<F32, 8>(wm);
    return nullptr;
}

}  // namespace rrn
