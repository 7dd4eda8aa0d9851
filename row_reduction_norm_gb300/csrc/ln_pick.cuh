// ln_pick.cuh -- maps runtime (threads per row, chunks, affine mode) to the
// compiled LayerNorm instantiations (internal).
#pragma once

#include "layernorm_kernels.cuh"

namespace rrn {
namespace lnpick {

template <typename T, int GT, int CH, bool RES>
const void *reg_aff(int aff) {
    switch (aff) {
        case kAffNone: return reinterpret_cast<const void *>(&ln_reg_kernel<T, GT, CH, RES, kAffNone>);
        case kAffW: return reinterpret_cast<const void *>(&ln_reg_kernel<T, GT, CH, RES, kAffW>);
        case kAffWB: return reinterpret_cast<const void *>(&ln_reg_kernel<T, GT, CH, RES, kAffWB>);
        default: return nullptr;
    }
}

template <typename T, int GT, bool RES>
const void *reg_ch(int ch, int aff) {
    switch (ch) {
        case 1: return reg_aff<T, GT, 1, RES>(aff);
        case 2: return reg_aff<T, GT, 2, RES>(aff);
        case 3: return reg_aff<T, GT, 3, RES>(aff);
        case 4: return reg_aff<T, GT, 4, RES>(aff);
        case 6: return reg_aff<T, GT, 6, RES>(aff);
        case 8: return reg_aff<T, GT, 8, RES>(aff);
        default: return nullptr;
    }
}

template <typename T, bool RES>
const void *reg_gt(int gt, int ch, int aff) {
    switch (gt) {
        case 4: return reg_ch<T, 4, RES>(ch, aff);
        case 8: return reg_ch<T, 8, RES>(ch, aff);
        case 16: return reg_ch<T, 16, RES>(ch, aff);
        case 32: return reg_ch<T, 32, RES>(ch, aff);
        case 64: return reg_ch<T, 64, RES>(ch, aff);
        case 128: return reg_ch<T, 128, RES>(ch, aff);
        case 256: return reg_ch<T, 256, RES>(ch, aff);
        default: return nullptr;
    }
}

template <typename T, int VE, int BLOCK, bool RES>
const void *loop_aff(int aff) {
    switch (aff) {
        case kAffNone: return reinterpret_cast<const void *>(&ln_loop_kernel<T, VE, BLOCK, RES, kAffNone>);
        case kAffW: return reinterpret_cast<const void *>(&ln_loop_kernel<T, VE, BLOCK, RES, kAffW>);
        case kAffWB: return reinterpret_cast<const void *>(&ln_loop_kernel<T, VE, BLOCK, RES, kAffWB>);
        default: return nullptr;
    }
}

template <typename T, bool RES>
const void *loop_block(int block, bool vec, int aff) {
    switch (block) {
        case 64: return vec ? loop_aff<T, T::kVec, 64, RES>(aff) : loop_aff<T, 1, 64, RES>(aff);
        case 256: return vec ? loop_aff<T, T::kVec, 256, RES>(aff) : loop_aff<T, 1, 256, RES>(aff);
        case 1024: return vec ? loop_aff<T, T::kVec, 1024, RES>(aff) : loop_aff<T, 1, 1024, RES>(aff);
        default: return nullptr;
    }
}

}  // namespace lnpick
}  // namespace rrn
