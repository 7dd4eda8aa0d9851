// layernorm_kernels.cuh -- sm_103a kernels of the fused row-wise LayerNorm.
//
// Per row: h = x (or RN_T(x + residual), stored as residual_out),
//   mu = mean(h), var = mean((h - mu)^2),
//   y  = RN_T( (h - mu) * rsqrt(var + eps) * w + b )      (w, b optional)
// Definition: "GPT-2 on the GPU", section "The Whole Model as One Kernel"
// (the traced GPT-2 block: mean, variance, (x - mean) / sqrt(var + eps),
// then weight * normalised + bias, eps 1e-5).
//
// The same two kernel shapes as the RMSNorm (see rmsnorm_kernels.cuh), with
// one more statistic:
//  * ln_reg_kernel: the row sits in registers, so the variance is taken in
//    an exact second pass over the centred values (no E[h^2] - mu^2
//    cancellation) at no extra memory traffic; two fixed-order reductions.
//  * ln_loop_kernel: rows not aligned to 16 bytes or too long for registers;
//    three passes (mean; centred squares; output), the second and third
//    reading the row back from L2.
// Fixed reduction order, no atomics: deterministic and batch-invariant.
#pragma once

#include "rmsnorm_kernels.cuh"

namespace rrn {

// Affine modes: none, weight only, weight and bias.
enum AffineMode { kAffNone = 0, kAffW = 1, kAffWB = 2 };

struct LnParams {
    const void *x;
    const void *res;     // nullable
    const void *w;       // nullable
    const void *b;       // nullable (requires w)
    void *y;
    void *res_out;       // nullable
    int64_t rows;
    int64_t row_elems;
    int64_t row_bytes;
    int32_t units;
    float hidden_f;
    float eps;
};

template <int AFF>
__device__ __forceinline__ float ln_out(float h, float mu, float r, float w, float b) {
    const float n = (h - mu) * r;
    if constexpr (AFF == kAffNone) {
        return n;
    } else if constexpr (AFF == kAffW) {
        return n * w;
    } else {
        return fmaf(n, w, b);
    }
}

// Block-wide combine of one fp32 value per row group (fixed order).  Uses
// red[parity] and flips parity; every thread of the row gets the same bits.
template <int LANES, int WPR, int RPB>
__device__ __forceinline__ float row_combine(float v, float (&red)[2][RPB][WPR], int &parity, int slot, int t,
                                             int tid) {
    v = butterfly_sum<LANES>(v);
    if constexpr (WPR > 1) {
        if ((tid & 31) == 0) red[parity][slot][t / 32] = v;
        __syncthreads();
        float s[WPR];
#pragma unroll
        for (int i = 0; i < WPR; ++i) s[i] = red[parity][slot][i];
        v = tree_sum(s);
        parity ^= 1;
    }
    return v;
}

// Threads per block of the LayerNorm register kernel: at least four warps
// (rows of a warp or less: 128 / threads_per_row rows a block).  Measured on
// GB300 against the RMSNorm kernel's 256: bf16 16384 x 768 with weight and
// bias 9.81 -> 9.52 us -- twice the blocks, so the last wave of each SM is
// half as coarse, for the same warps resident.
__host__ __device__ constexpr int ln_block_threads(int gt) { return gt >= 128 ? gt : 128; }

// Resident 256-thread equivalents the register budget is sized for: four (64
// registers a thread) for up to 4 chunks a thread, which keeps enough loads in
// flight per SM; five (48 registers) for up to 3 chunks without a residual,
// which fit them without spilling (measured on GB300: bf16 16384 x 768 with
// weight and bias 11.47 -> 10.65 us; six spill and are slower); two (128
// registers) for 8 chunks.  Blocks of 128 threads get twice as many.
__host__ __device__ constexpr int ln_min_blocks(int gt, int ch, bool res) {
    return (ln_block_threads(gt) == 128 ? 2 : 1) * ((ch <= 3 && !res) ? 5 : (ch <= 4 ? 4 : 2));
}

template <typename T, int GT, int CH, bool RES, int AFF>
__global__ void __launch_bounds__(ln_block_threads(GT), ln_min_blocks(GT, CH, RES))
ln_reg_kernel(const LnParams p) {
    constexpr int V = T::kVec;
    constexpr int BLOCK = ln_block_threads(GT);
    constexpr int RPB = BLOCK / GT;
    constexpr int LANES = GT < 32 ? GT : 32;
    constexpr int WPR = GT > 32 ? GT / 32 : 1;
    constexpr bool W = AFF != kAffNone;
    constexpr bool B = AFF == kAffWB;
    static_assert((GT & (GT - 1)) == 0 && GT >= 4 && GT <= 1024, "GT: power of two in [4, 1024]");
    __shared__ float red[2][RPB][WPR];

    const int tid = threadIdx.x;
    const int slot = tid / GT;
    const int t = tid % GT;
    const int nch = p.units;

    // before the wait: the block's first row group into L2 (see prefetch_rows_l2)
    if (tid == 0) prefetch_rows_l2<RES>(p.x, p.res, p.row_bytes, p.rows, (int64_t)blockIdx.x * RPB, RPB);
    pdl_wait_for_inputs();
    pdl_allow_dependents();

    // w (and b) staged once per block in shared memory: [w chunks | b chunks]
    extern __shared__ Chunk wb_smem[];
    bool staged = false;
    int parity = 0;

    for (int64_t rb = blockIdx.x; rb * RPB < p.rows; rb += gridDim.x) {
        const int64_t row = rb * RPB + slot;
        const bool row_ok = row < p.rows;
        const int64_t off = row_ok ? row * p.row_bytes : 0;

        // the row's chunks (zeros past the row end)
        Chunk hc[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int u = c * GT + t;
            if (row_ok && u < nch)
                hc[c] = ld_stream16(static_cast<const char *>(p.x) + off + (int64_t)u * 16);
            else
                hc[c] = Chunk{{0u, 0u, 0u, 0u}};
        }
        Chunk rc[RES ? CH : 1];
        if constexpr (RES) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int u = c * GT + t;
                if (row_ok && u < nch)
                    rc[c] = ld_stream16(static_cast<const char *>(p.res) + off + (int64_t)u * 16);
                else
                    rc[c] = Chunk{{0u, 0u, 0u, 0u}};
            }
        }
        if constexpr (W) {
            if (!staged) {   // first iteration of the block (uniform across it)
                for (int i = tid; i < nch; i += BLOCK)
                    wb_smem[i] = ld_readonly16(static_cast<const char *>(p.w) + (int64_t)i * 16);
                if constexpr (B) {
                    for (int i = tid; i < nch; i += BLOCK)
                        wb_smem[nch + i] = ld_readonly16(static_cast<const char *>(p.b) + (int64_t)i * 16);
                }
                __syncthreads();
                staged = true;
            }
        }
        if constexpr (RES) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int u = c * GT + t;
                float a[V], bb[V];
                unpack(hc[c], a, T{});
                unpack(rc[c], bb, T{});
#pragma unroll
                for (int e = 0; e < V; ++e) a[e] = add_round(a[e], bb[e], T{});
                hc[c] = pack(a, T{});
                if (row_ok && u < nch)
                    st16(static_cast<char *>(p.res_out) + off + (int64_t)u * 16, hc[c]);
            }
        }
        // mean: sum in V accumulators, chunk order, fixed tree
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            float a[V];
            unpack(hc[c], a, T{});
            add_pairs(acc, a);
        }
        const float mu = row_combine<LANES, WPR, RPB>(tree_sum(acc), red, parity, slot, t, tid) / p.hidden_f;
        // variance: centred squares of the valid elements (slots past the row end are skipped)
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
        const float2 nmu2 = make_float2(-mu, -mu);
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int u = c * GT + t;
            if (u < nch) {
                float a[V];
                unpack(hc[c], a, T{});
#pragma unroll
                for (int k = 0; k < V / 2; ++k) {
                    const float2 d = __fadd2_rn(make_float2(a[2 * k], a[2 * k + 1]), nmu2);
                    const float2 q = __ffma2_rn(d, d, make_float2(acc[2 * k], acc[2 * k + 1]));
                    acc[2 * k] = q.x;
                    acc[2 * k + 1] = q.y;
                }
            }
        }
        const float var = row_combine<LANES, WPR, RPB>(tree_sum(acc), red, parity, slot, t, tid) / p.hidden_f;
        const float r = rsqrtf(var + p.eps);
        const float2 r2 = make_float2(r, r);
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int u = c * GT + t;
            if (row_ok && u < nch) {
                float a[V], wv[V], bv[V];
                unpack(hc[c], a, T{});
                if constexpr (W) unpack(wb_smem[u], wv, T{});
                if constexpr (B) unpack(wb_smem[nch + u], bv, T{});
#pragma unroll
                for (int k = 0; k < V / 2; ++k) {
                    // n = (h - mu) * r, then n * w or fma(n, w, b): two lanes at a time
                    float2 n = __fmul2_rn(__fadd2_rn(make_float2(a[2 * k], a[2 * k + 1]), nmu2), r2);
                    if constexpr (AFF == kAffW) {
                        n = __fmul2_rn(n, make_float2(wv[2 * k], wv[2 * k + 1]));
                    } else if constexpr (AFF == kAffWB) {
                        n = __ffma2_rn(n, make_float2(wv[2 * k], wv[2 * k + 1]), make_float2(bv[2 * k], bv[2 * k + 1]));
                    }
                    a[2 * k] = n.x;
                    a[2 * k + 1] = n.y;
                }
                st16(static_cast<char *>(p.y) + off + (int64_t)u * 16, pack(a, T{}));
            }
        }
    }
}

template <typename T, int VE, int BLOCK, bool RES, int AFF>
__global__ void __launch_bounds__(BLOCK, 1)
ln_loop_kernel(const LnParams p) {
    using IO = UnitIO<T, VE>;
    using Raw = typename IO::Raw;
    constexpr int NACC = 8;
    constexpr int U = VE == 1 ? NACC : 2;
    constexpr int NW = BLOCK / 32;
    constexpr bool W = AFF != kAffNone;
    constexpr bool B = AFF == kAffWB;
    static_assert(BLOCK % 32 == 0 && (NW & (NW - 1)) == 0, "BLOCK: power-of-two warps");
    __shared__ float red[2][1][NW];

    const int tid = threadIdx.x;
    const int64_t nunits = p.units;
    int parity = 0;
    pdl_wait_for_inputs();
    pdl_allow_dependents();

    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const int64_t off = row * p.row_bytes;
        const void *xr = static_cast<const char *>(p.x) + off;
        const void *rr = RES ? static_cast<const char *>(p.res) + off : nullptr;
        void *hr = RES ? static_cast<char *>(p.res_out) + off : nullptr;
        void *yr = static_cast<char *>(p.y) + off;
        const void *src = RES ? static_cast<const void *>(hr) : xr;

        // pass 1: h (and residual_out), sum
        float acc[NACC];
#pragma unroll
        for (int i = 0; i < NACC; ++i) acc[i] = 0.f;
        for (int64_t base = tid; base < nunits; base += (int64_t)BLOCK * U) {
            Raw xa[U];
            Raw rb[RES ? U : 1];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t u = base + (int64_t)j * BLOCK;
                xa[j] = u < nunits ? IO::load_first(xr, u) : IO::zero();
            }
            if constexpr (RES) {
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const int64_t u = base + (int64_t)j * BLOCK;
                    rb[j] = u < nunits ? IO::load_first(rr, u) : IO::zero();
                }
            }
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t u = base + (int64_t)j * BLOCK;
                float a[VE];
                IO::widen(xa[j], a);
                if constexpr (RES) {
                    float bb[VE];
                    IO::widen(rb[j], bb);
#pragma unroll
                    for (int e = 0; e < VE; ++e) a[e] = add_round(a[e], bb[e], T{});
                    if (u < nunits) IO::store(hr, u, a);
                }
#pragma unroll
                for (int e = 0; e < VE; ++e) acc[(j * VE + e) % NACC] += a[e];
            }
        }
        const float mu = row_combine<32, NW, 1>(tree_sum(acc), red, parity, 0, tid, tid) / p.hidden_f;

        // pass 2: centred squares (row read back from L2)
#pragma unroll
        for (int i = 0; i < NACC; ++i) acc[i] = 0.f;
        for (int64_t base = tid; base < nunits; base += (int64_t)BLOCK * U) {
            Raw ha[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t u = base + (int64_t)j * BLOCK;
                ha[j] = u < nunits ? IO::load_first(src, u) : IO::zero();
            }
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t u = base + (int64_t)j * BLOCK;
                if (u < nunits) {
                    float a[VE];
                    IO::widen(ha[j], a);
#pragma unroll
                    for (int e = 0; e < VE; ++e) {
                        const float d = a[e] - mu;
                        const int k = (j * VE + e) % NACC;
                        acc[k] = fmaf(d, d, acc[k]);
                    }
                }
            }
        }
        const float var = row_combine<32, NW, 1>(tree_sum(acc), red, parity, 0, tid, tid) / p.hidden_f;
        const float r = rsqrtf(var + p.eps);

        // pass 3: output
        for (int64_t base = tid; base < nunits; base += (int64_t)BLOCK * U) {
            Raw ha[U];
            Raw wa[W ? U : 1];
            Raw ba[B ? U : 1];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t u = base + (int64_t)j * BLOCK;
                ha[j] = u < nunits ? IO::load_last(src, u) : IO::zero();
                if constexpr (W) wa[j] = u < nunits ? IO::load_w(p.w, u) : IO::zero();
                if constexpr (B) ba[j] = u < nunits ? IO::load_w(p.b, u) : IO::zero();
            }
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t u = base + (int64_t)j * BLOCK;
                float a[VE], wv[VE], bv[VE];
                IO::widen(ha[j], a);
                if constexpr (W) IO::widen(wa[j], wv);
                if constexpr (B) IO::widen(ba[j], bv);
#pragma unroll
                for (int e = 0; e < VE; ++e)
                    a[e] = ln_out<AFF>(a[e], mu, r, W ? wv[e] : 1.f, B ? bv[e] : 0.f);
                if (u < nunits) IO::store(yr, u, a);
            }
        }
    }
}

}  // namespace rrn
