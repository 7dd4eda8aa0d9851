// kernel_pick.cuh -- maps runtime (threads per row, chunks, weight mode) to
// compiled instantiations (internal; included by the instantiation files).
#pragma once

#include <type_traits>

#include "rmsnorm_kernels.cuh"

namespace rrn {
namespace pick {

// CAST instantiates only the cast-order weight mode (bf16 contiguous rows, in
// a translation unit of its own); otherwise the three plain modes.
template <typename T, int GT, int CH, bool RES, bool HEADS, bool CAST>
const void *reg_wm(int wm) {
    if constexpr (CAST) {
        static_assert(!HEADS && std::is_same<T, BF16>::value, "cast order: bf16 contiguous rows");
        return wm == kWeightCast ? reinterpret_cast<const void *>(&rms_reg_kernel<T, GT, CH, RES, kWeightCast, false>)
                                 : nullptr;
    } else {
        switch (wm) {
            case kNoWeight: return reinterpret_cast<const void *>(&rms_reg_kernel<T, GT, CH, RES, kNoWeight, HEADS>);
            case kWeight: return reinterpret_cast<const void *>(&rms_reg_kernel<T, GT, CH, RES, kWeight, HEADS>);
            case kWeightBias:
                return reinterpret_cast<const void *>(&rms_reg_kernel<T, GT, CH, RES, kWeightBias, HEADS>);
            default: return nullptr;
        }
    }
}

// Chunks per thread: powers of two, plus 3 and 6 for contiguous rows (rows of
// 3 * 2^k or 6 * 2^k chunks, e.g. widths 576 and 768, then fill every slot).
template <typename T, int GT, bool RES, bool HEADS, bool CAST = false>
const void *reg_ch(int ch, int wm) {
    switch (ch) {
        case 1: return reg_wm<T, GT, 1, RES, HEADS, CAST>(wm);
        case 2: return reg_wm<T, GT, 2, RES, HEADS, CAST>(wm);
        case 4: return reg_wm<T, GT, 4, RES, HEADS, CAST>(wm);
        case 8: return reg_wm<T, GT, 8, RES, HEADS, CAST>(wm);
        default: break;
    }
    if constexpr (!HEADS) {
        switch (ch) {
            case 3: return reg_wm<T, GT, 3, RES, HEADS, CAST>(wm);
            case 6: return reg_wm<T, GT, 6, RES, HEADS, CAST>(wm);
            default: break;
        }
    }
    return nullptr;
}

template <typename T, bool RES, bool HEADS, int MAXGT, bool CAST = false>
const void *reg_gt(int gt, int ch, int wm) {
    switch (gt) {
        case 4: return reg_ch<T, 4, RES, HEADS, CAST>(ch, wm);
        case 8: return reg_ch<T, 8, RES, HEADS, CAST>(ch, wm);
        case 16: return reg_ch<T, 16, RES, HEADS, CAST>(ch, wm);
        case 32: return reg_ch<T, 32, RES, HEADS, CAST>(ch, wm);
        default: break;
    }
    if constexpr (MAXGT >= 512) {
        switch (gt) {
            case 64: return reg_ch<T, 64, RES, HEADS, CAST>(ch, wm);
            case 128: return reg_ch<T, 128, RES, HEADS, CAST>(ch, wm);
            case 256: return reg_ch<T, 256, RES, HEADS, CAST>(ch, wm);
            case 512: return reg_ch<T, 512, RES, HEADS, CAST>(ch, wm);
            default: break;
        }
    }
    return nullptr;
}

// MXFP8 output (contiguous rows; at least 32 / V lanes per row).
template <typename T, int GT, int CH, bool RES>
const void *mx_wm(int wm) {
    switch (wm) {
        case kNoWeight: return reinterpret_cast<const void *>(&rms_quant_kernel<T, GT, CH, RES, kNoWeight, kOutMxfp8>);
        case kWeight: return reinterpret_cast<const void *>(&rms_quant_kernel<T, GT, CH, RES, kWeight, kOutMxfp8>);
        case kWeightBias:
            return reinterpret_cast<const void *>(&rms_quant_kernel<T, GT, CH, RES, kWeightBias, kOutMxfp8>);
        default: return nullptr;
    }
}

template <typename T, int GT, bool RES>
const void *mx_ch(int ch, int wm) {
    if constexpr (GT < 32 / T::kVec) {
        return nullptr;
    } else {
        switch (ch) {
            case 1: return mx_wm<T, GT, 1, RES>(wm);
            case 2: return mx_wm<T, GT, 2, RES>(wm);
            case 4: return mx_wm<T, GT, 4, RES>(wm);
            case 8: return mx_wm<T, GT, 8, RES>(wm);
            default: return nullptr;
        }
    }
}

template <typename T, bool RES>
const void *mx_gt(int gt, int ch, int wm) {
    switch (gt) {
        case 4: return mx_ch<T, 4, RES>(ch, wm);
        case 8: return mx_ch<T, 8, RES>(ch, wm);
        case 16: return mx_ch<T, 16, RES>(ch, wm);
        case 32: return mx_ch<T, 32, RES>(ch, wm);
        case 64: return mx_ch<T, 64, RES>(ch, wm);
        case 128: return mx_ch<T, 128, RES>(ch, wm);
        case 256: return mx_ch<T, 256, RES>(ch, wm);
        case 512: return mx_ch<T, 512, RES>(ch, wm);
        default: return nullptr;
    }
}

// NVFP4 output (contiguous rows).
template <typename T, int GT, int CH, bool RES>
const void *nv_wm(int wm) {
    switch (wm) {
        case kNoWeight: return reinterpret_cast<const void *>(&rms_quant_kernel<T, GT, CH, RES, kNoWeight, kOutNvfp4>);
        case kWeight: return reinterpret_cast<const void *>(&rms_quant_kernel<T, GT, CH, RES, kWeight, kOutNvfp4>);
        case kWeightBias:
            return reinterpret_cast<const void *>(&rms_quant_kernel<T, GT, CH, RES, kWeightBias, kOutNvfp4>);
        default: return nullptr;
    }
}

template <typename T, int GT, bool RES>
const void *nv_ch(int ch, int wm) {
    switch (ch) {
        case 1: return nv_wm<T, GT, 1, RES>(wm);
        case 2: return nv_wm<T, GT, 2, RES>(wm);
        case 4: return nv_wm<T, GT, 4, RES>(wm);
        case 8: return nv_wm<T, GT, 8, RES>(wm);
        default: return nullptr;
    }
}

template <typename T, bool RES>
const void *nv_gt(int gt, int ch, int wm) {
    switch (gt) {
        case 4: return nv_ch<T, 4, RES>(ch, wm);
        case 8: return nv_ch<T, 8, RES>(ch, wm);
        case 16: return nv_ch<T, 16, RES>(ch, wm);
        case 32: return nv_ch<T, 32, RES>(ch, wm);
        case 64: return nv_ch<T, 64, RES>(ch, wm);
        case 128: return nv_ch<T, 128, RES>(ch, wm);
        case 256: return nv_ch<T, 256, RES>(ch, wm);
        case 512: return nv_ch<T, 512, RES>(ch, wm);
        default: return nullptr;
    }
}

template <typename T, int VE, int BLOCK, bool RES, bool HEADS, bool CAST>
const void *loop_wm(int wm) {
    if constexpr (CAST) {
        static_assert(!HEADS && std::is_same<T, BF16>::value, "cast order: bf16 contiguous rows");
        return wm == kWeightCast
                   ? reinterpret_cast<const void *>(&rms_loop_kernel<T, VE, BLOCK, RES, kWeightCast, false>)
                   : nullptr;
    } else {
        switch (wm) {
            case kNoWeight:
                return reinterpret_cast<const void *>(&rms_loop_kernel<T, VE, BLOCK, RES, kNoWeight, HEADS>);
            case kWeight: return reinterpret_cast<const void *>(&rms_loop_kernel<T, VE, BLOCK, RES, kWeight, HEADS>);
            case kWeightBias:
                return reinterpret_cast<const void *>(&rms_loop_kernel<T, VE, BLOCK, RES, kWeightBias, HEADS>);
            default: return nullptr;
        }
    }
}

template <typename T, bool RES, bool HEADS, bool CAST = false>
const void *loop_block(int block, bool vec, int wm) {
    switch (block) {
        case 64: return vec ? loop_wm<T, T::kVec, 64, RES, HEADS, CAST>(wm) : loop_wm<T, 1, 64, RES, HEADS, CAST>(wm);
        case 256: return vec ? loop_wm<T, T::kVec, 256, RES, HEADS, CAST>(wm) : loop_wm<T, 1, 256, RES, HEADS, CAST>(wm);
        case 1024: return vec ? loop_wm<T, T::kVec, 1024, RES, HEADS, CAST>(wm) : loop_wm<T, 1, 1024, RES, HEADS, CAST>(wm);
        default: return nullptr;
    }
}

}  // namespace pick
}  // namespace rrn
