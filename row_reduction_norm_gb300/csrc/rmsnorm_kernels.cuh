// rmsnorm_kernels.cuh -- sm_103a kernels of the fused row-wise RMSNorm.
//
// The op, per row: h = x (or RN_T(x + residual), stored as residual_out),
// y = RN_T(h * rsqrt(mean(h^2) + eps) * w).  Definition: "Building a GPU
// compiler from scratch: from PyTorch to CUDA via multi-level IR (Emmy)",
// running example and section "Tensor IR" (square, sum, division by the count,
// plus epsilon, rsqrt, two multiplications); section "Loop IR" fuses all of it
// into one kernel whose statistic never leaves the chip, which is what both
// kernel families below do.
//
// This path is a row reduction bound by HBM bandwidth (about 1 flop per byte),
// not a contraction, so it uses no tensor cores.  What matters on GB300 is
// bytes in flight per SM, coalesced 128-bit accesses and a grid sized to the
// SM count:
//
//  * rms_reg_kernel  -- the row lives in registers.  threads_per_row (GT)
//    threads cooperate on a row, each owning up to CH 16-byte chunks
//    (chunk index c*GT + t), so a warp's loads of one chunk slot cover 32
//    consecutive 16-byte pieces.  GT <= 32 is the warp / sub-warp regime
//    ("CuTeDSL at Perplexity", section "QK Norm": a half warp of 16 lanes x 8
//    bf16 covers a 128-element head, reduced with xor butterflies); GT > 32
//    adds a shared-memory combine across the row's warps (the "256 workers
//    per row" schedule of the Emmy page, section "Tile IR").  Blocks stride
//    over row groups, so a grid capped at the resident capacity is the
//    persistent regime.  w (the same for every row) is loaded by each lane
//    next to its x chunks when a row is at most a warp (L1 serves the
//    block's other rows), and staged once per block in shared memory when a
//    row spans several warps or the output is block-scaled.
//  * Both kernels also serve head rows (the fused Q+K norm of the Perplexity
//    page's "QK Norm" section): rows are the heads of each token inside a
//    packed projection, and query and key heads take different weights.
//  * rms_loop_kernel -- one block per row, the row streamed twice: the first
//    pass forms h (and writes residual_out) and the sum of squares, the second
//    re-reads h (an L2 hit: the rows in flight are far smaller than L2) and
//    writes y.  It serves rows whose pointers are not 16-byte aligned
//    (scalar accesses) and rows too long to hold in registers.
//
// Reduction order is fixed by (hidden, dtype, alignment) alone: per-thread
// accumulators in a set order, a fixed tree over them, xor butterflies, then
// a fixed tree over warps.  No atomics.  A row's result therefore does not
// depend on the row count or grid, and repeated runs are bit-identical
// (the determinism requirement of the model-as-a-kernel card).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rrn {

// Kernel arguments (passed by value).
//
// Row addressing.  Contiguous rows: row r starts x_stride * r bytes into x
// (residual shares x's layout) and y_stride * r bytes into y (residual_out
// shares y's).  Head rows (the fused Q+K norm): row r is head j = r % heads of
// token t = r / heads, at t * x_stride + j * row_bytes in x and likewise in y;
// heads j < q_heads take weight w, the others w2.
struct Params {
    const void *x;
    const void *res;     // nullable
    const void *w;       // nullable
    const void *w2;      // second weight (head rows: the key heads' weight)
    void *y;
    void *res_out;       // nullable
    int64_t rows;        // rows, or tokens * heads
    int64_t row_elems;   // elements per row (hidden or head_dim)
    int64_t row_bytes;   // row_elems * sizeof(T)
    int64_t x_stride;    // bytes between consecutive rows (tokens for head rows) of x
    int64_t y_stride;    // same for y
    int32_t units;       // loads per row: row_elems / vec_elems
    int32_t heads;       // heads per token (head rows), else 1
    int32_t q_heads;     // heads per token that take w
    float hidden_f;      // row_elems as float (exact for row_elems <= 2^24)
    float eps;
    float w_bias;        // added to every weight element (weight mode kWeightBias)
    void *scales;        // block-scaled outputs: the scales (y holds the codes)
    float q_scale;       // NVFP4: per-tensor scale S
    float q_inv6s;       // NVFP4: 1 / (6 S), rounded once to float
    int32_t rpb;         // register kernel: rows a block holds per iteration
                         // (BLOCK / GT, or fewer for a launch of few rows)
    uint64_t wait_ns;    // bulk-copy kernel: limit of each of its waits, in ns
    int32_t withhold;    // bulk-copy kernel, tests of its bounded waits only:
                         // 1 = block 0's first consumer warp keeps its first
                         // x slot (0 in every library launch)
};

// Output form of the register kernel: the I/O type; MXFP8 (E4M3 codes in y,
// one E8M0 scale per 32 elements in scales); NVFP4 (E2M1 codes packed two a
// byte in y, one E4M3 scale per 16 elements in scales).
enum OutputMode { kOutT = 0, kOutMxfp8 = 1, kOutNvfp4 = 2 };

// How the weight enters y: none, w, (w + w_bias), or w after the normalised
// value has been rounded to bf16 (the op-by-op cast order of an eager
// framework, "model-as-a-kernel", sections "Method" and "Correctness"; bf16
// I/O only, since with fp32 I/O the kWeight product is already rounded to the
// I/O type before the weight multiply).
enum WeightMode { kNoWeight = 0, kWeight = 1, kWeightBias = 2, kWeightCast = 3 };

template <int WM>
__device__ __forceinline__ float scale_out(float h, float r, float w, float bias) {
    if constexpr (WM == kNoWeight) {
        return h * r;
    } else if constexpr (WM == kWeight) {
        return (h * r) * w;
    } else if constexpr (WM == kWeightCast) {
        return __bfloat162float(__float2bfloat16_rn(h * r)) * w;
    } else {
        return (h * r) * (w + bias);
    }
}

// Byte offsets of row `row` in x and y, and which weight it takes.
template <bool HEADS>
__device__ __forceinline__ void row_offsets(const Params &p, int64_t row, int64_t &xo, int64_t &yo, int &wsel) {
    if constexpr (HEADS) {
        const int64_t tok = row / p.heads;
        const int j = (int)(row - tok * p.heads);
        const int64_t hoff = (int64_t)j * p.row_bytes;
        xo = tok * p.x_stride + hoff;
        yo = tok * p.y_stride + hoff;
        wsel = j >= p.q_heads ? 1 : 0;
    } else {
        xo = row * p.x_stride;
        yo = row * p.y_stride;
        wsel = 0;
    }
}

struct BF16 {
    using storage = uint16_t;
    static constexpr int kVec = 8;   // elements per 16-byte chunk
};
struct F32 {
    using storage = float;
    static constexpr int kVec = 4;
};

struct __align__(16) Chunk {
    uint32_t u[4];
};

// ------------------------------------------------------------------ memory
// x and residual are read once: keep them out of L1 and mark their L2 lines
// first to go.  w is read-only and reused by every row: the read-only path.
// Plain (not .nc) loads for x/residual keep in-place calls (y == x) safe.

__device__ __forceinline__ Chunk ld_stream16(const void *p) {
    Chunk c;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(c.u[0]), "=r"(c.u[1]), "=r"(c.u[2]), "=r"(c.u[3])
                 : "l"(p));
    return c;
}

// First read of a row that will be read again from L2 (two-pass kernel).
__device__ __forceinline__ Chunk ld_keep_l2_16(const void *p) {
    Chunk c;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(c.u[0]), "=r"(c.u[1]), "=r"(c.u[2]), "=r"(c.u[3])
                 : "l"(p));
    return c;
}

__device__ __forceinline__ Chunk ld_readonly16(const void *p) {
    Chunk c;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(c.u[0]), "=r"(c.u[1]), "=r"(c.u[2]), "=r"(c.u[3])
                 : "l"(p));
    return c;
}

__device__ __forceinline__ void st16(void *p, const Chunk &c) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :
                 : "l"(p), "r"(c.u[0]), "r"(c.u[1]), "r"(c.u[2]), "r"(c.u[3])
                 : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the kernel before it drains.  It must not
// read its inputs before griddepcontrol.wait returns (the grids it depends on
// have completed and their writes are visible); without that launch
// attribute the wait returns at once.  Signalling launch_dependents at entry
// lets the next kernel's blocks be placed as soon as every block of this one
// is resident.
__device__ __forceinline__ void pdl_wait_for_inputs() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// L2 prefetch of `bytes` bytes at `p` (16-byte aligned, a multiple of 16 bytes)
// through the bulk-copy engine.  It returns no data to the thread and fills no
// L1 line; it only warms L2, which is the device's point of coherence for
// global memory.  So it may be issued before griddepcontrol.wait, even on
// memory the kernel still running ahead of this one is writing: every load
// of the kernel comes after the wait, reads the line in L2, and sees the
// earlier kernel's stores there (a line prefetched before a store is updated
// by that store).  A prefetch changes timing, never a value.
__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" : : "l"(p), "r"(bytes) : "memory");
}

// The first rows a block will read (rows r0 .. r0 + n - 1 of contiguous
// [rows, row_bytes] tensors x and, with RES, the residual), prefetched into
// L2 by the calling thread before the block waits on the kernel ahead of it.
// Measured on GB300: a launch whose inputs were not written by the kernel
// just before it (the residual stream of a transformer block, or any norm
// after an unrelated kernel) saves one DRAM round trip of its critical path
// -- bf16 4096 x 576 3.03 -> 2.24 us a launch, decode 1 x 4096 1.74 -> 1.47
// us; when the kernel before it has just written x the lines are already in
// L2 and the launch costs the same (2.158 -> 2.159 us).  A weight prefetched
// the same way measured slower (it is read by every block and stays in L2).
template <bool RES>
__device__ __forceinline__ void prefetch_rows_l2(const void *x, const void *res, int64_t row_bytes, int64_t rows,
                                                 int64_t r0, int n) {
    if (r0 >= rows) return;
    const int64_t nr = rows - r0 < n ? rows - r0 : n;
    const unsigned bytes = (unsigned)(nr * row_bytes);
    prefetch_l2(static_cast<const char *>(x) + r0 * row_bytes, bytes);
    if constexpr (RES) prefetch_l2(static_cast<const char *>(res) + r0 * row_bytes, bytes);
}

// ------------------------------------------------------------- conversions
// bf16 is the upper half of an fp32 encoding: widening is a 16-bit shift.
// Narrowing rounds to nearest even with the CUDA intrinsic.

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);   // .x = lo (lower address)
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ void unpack(const Chunk &c, float (&f)[8], BF16) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = bf16_lo(c.u[k]);
        f[2 * k + 1] = bf16_hi(c.u[k]);
    }
}
__device__ __forceinline__ void unpack(const Chunk &c, float (&f)[4], F32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) f[k] = __uint_as_float(c.u[k]);
}
__device__ __forceinline__ Chunk pack(const float (&f)[8], BF16) {
    Chunk c;
#pragma unroll
    for (int k = 0; k < 4; ++k) c.u[k] = pack_bf16x2(f[2 * k], f[2 * k + 1]);
    return c;
}
__device__ __forceinline__ Chunk pack(const float (&f)[4], F32) {
    Chunk c;
#pragma unroll
    for (int k = 0; k < 4; ++k) c.u[k] = __float_as_uint(f[k]);
    return c;
}

// RN_T(a + b) for the residual add: one fp32 add, then one rounding to T.
// For bf16 the fp32 sum of two bf16 values rounded to bf16 equals the
// correctly rounded sum (fp32 carries more than 2*8+2 significant bits).
__device__ __forceinline__ float add_round(float a, float b, BF16) {
    return __bfloat162float(__float2bfloat16_rn(__fadd_rn(a, b)));
}
__device__ __forceinline__ float add_round(float a, float b, F32) { return __fadd_rn(a, b); }

// ------------------------------------------------------- packed fp32 math
// sm_100+ issues two fp32 operations per instruction on register pairs
// (FFMA2 / FMUL2 / FADD2).  Each half rounds exactly as the scalar operation
// does, so these helpers change instruction counts, not results.

template <int N>
__device__ __forceinline__ void sq_accumulate(const float (&a)[N], float (&acc)[N]) {
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
        const float2 v = make_float2(a[2 * k], a[2 * k + 1]);
        const float2 r = __ffma2_rn(v, v, make_float2(acc[2 * k], acc[2 * k + 1]));
        acc[2 * k] = r.x;
        acc[2 * k + 1] = r.y;
    }
}

template <int N>
__device__ __forceinline__ void add_pairs(float (&acc)[N], const float (&a)[N]) {
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
        const float2 r = __fadd2_rn(make_float2(acc[2 * k], acc[2 * k + 1]), make_float2(a[2 * k], a[2 * k + 1]));
        acc[2 * k] = r.x;
        acc[2 * k + 1] = r.y;
    }
}

// a[e] = scale_out<WM>(a[e], r, w[e], bias) for every e, two lanes at a time.
template <int WM, int N>
__device__ __forceinline__ void scale_out_pairs(float (&a)[N], float r, const float (&w)[N], float bias) {
    const float2 r2 = make_float2(r, r);
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
        float2 v = __fmul2_rn(make_float2(a[2 * k], a[2 * k + 1]), r2);
        if constexpr (WM == kWeight) {
            v = __fmul2_rn(v, make_float2(w[2 * k], w[2 * k + 1]));
        } else if constexpr (WM == kWeightCast) {
            v = __bfloat1622float2(__float22bfloat162_rn(v));   // exact product below: 8 x 8 bits
            v = __fmul2_rn(v, make_float2(w[2 * k], w[2 * k + 1]));
        } else if constexpr (WM == kWeightBias) {
            const float2 wb = __fadd2_rn(make_float2(w[2 * k], w[2 * k + 1]), make_float2(bias, bias));
            v = __fmul2_rn(v, wb);
        }
        a[2 * k] = v.x;
        a[2 * k + 1] = v.y;
    }
}

// ----------------------------------------------------------------- helpers

__host__ __device__ constexpr int reg_block_threads(int gt) { return gt >= 256 ? gt : 256; }

template <int LANES>
__device__ __forceinline__ float butterfly_sum(float v) {
    // xor butterfly inside aligned groups of LANES lanes; a + b == b + a, so
    // every lane of a group ends with the same bits.
#pragma unroll
    for (int off = LANES / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

template <int N>
__device__ __forceinline__ float tree_sum(float (&v)[N]) {
#pragma unroll
    for (int s = N / 2; s > 0; s >>= 1) {
#pragma unroll
        for (int i = 0; i < s; ++i) v[i] += v[i + s];
    }
    return v[0];
}

// ------------------------------------------------------- register kernel

// MXFP8 (OCP Microscaling v1.0, E4M3 elements): a block of 32 consecutive
// elements of a row shares the scale 2^s, s = floor(log2(amax)) - 8 clamped
// to [-127, 127] (-127 for an all-zero block); elements are E4M3 of v / 2^s,
// nearest-even, saturated at 448.  A block holding NaN or Inf is all NaN
// (scale 0xFF, codes 0x7F).  With the row's chunk c*GT + t owned by thread
// t, the 32 elements of a block sit in LPB = 32 / V consecutive lanes, which
// combine their maxima with xor shuffles.  The maxima propagate NaN
// (max.NaN), so a block's maximum is NaN or Inf exactly when one of its
// elements is: that one value marks the special blocks.
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

template <int LPB>
__device__ __forceinline__ float block_amax(float amax) {
#pragma unroll
    for (int off = LPB / 2; off > 0; off >>= 1) amax = max_nan(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    return amax;
}

// E8M0 exponent of a block from its (finite, non-negative) amax.
__device__ __forceinline__ int mx_scale_exponent(float amax) {
    const int ef = (__float_as_int(amax) >> 23) & 0xFF;   // 0: zero or subnormal
    const int s = ef == 0 ? -127 : ef - 127 - 8;
    return s < -127 ? -127 : s;
}

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// NVFP4: a block of 16 consecutive elements of a row (16 / V lanes) takes the
// scale E4M3(amax / (6 S)) (nearest-even, saturating) and the codes
// E2M1(v / (scale * S)), nearest-even, saturated at 6, two per byte with the
// even element in the low nibble; codes are 0 when the scale is 0.  A block
// holding NaN or Inf gets the E4M3 NaN 0x7F as its scale and codes 0.
__device__ __forceinline__ uint8_t e4m3_of(float v) {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// Value of a finite E4M3 code: the hardware conversion to fp16 (every E4M3
// value is exact in fp16), then to fp32.
__device__ __forceinline__ float e4m3_value(uint8_t c) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3)));
}

__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest);
}

// A7, block-scaled forms: the fp32 values a[] (h * r * w, not rounded) of
// chunk u of `row`, quantised with the other lanes of their block and stored
// (codes, and the block's scale from its first lane).  Every lane of a block
// calls it together, with the same `valid`; t is the thread's index in the
// row's group of threads.
template <int V, int OUT>
__device__ __forceinline__ void store_quantised(float (&a)[V], bool valid, const Params &p, int64_t row, int u,
                                                int t) {
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < V; ++e) amax = max_nan(amax, fabsf(a[e]));
    if constexpr (OUT == kOutMxfp8) {
        constexpr int LPB = 32 / V;
        amax = block_amax<LPB>(amax);
        const bool special = !(amax <= 3.402823466e38f);     // NaN or Inf in the block
        const int s = mx_scale_exponent(amax);
        const float mult = __int_as_float((127 - s) << 23);   // 2^-s, a normal float
        uint32_t q[V / 4];
#pragma unroll
        for (int k = 0; k < V / 4; ++k) {
            const uint32_t lo = e4m3x2(a[4 * k] * mult, a[4 * k + 1] * mult);
            const uint32_t hi = e4m3x2(a[4 * k + 2] * mult, a[4 * k + 3] * mult);
            q[k] = special ? 0x7F7F7F7Fu : (lo | (hi << 16));
        }
        if (valid) {
            char *dst = static_cast<char *>(p.y) + row * p.row_elems + (int64_t)u * V;
            if constexpr (V == 8) {
                asm volatile("st.global.v2.u32 [%0], {%1, %2};" : : "l"(dst), "r"(q[0]), "r"(q[1]) : "memory");
            } else {
                asm volatile("st.global.u32 [%0], %1;" : : "l"(dst), "r"(q[0]) : "memory");
            }
            if (t % LPB == 0) {
                const uint8_t sc = special ? (uint8_t)0xFF : (uint8_t)(s + 127);
                static_cast<uint8_t *>(p.scales)[row * (p.row_elems / 32) + u / LPB] = sc;
            }
        }
    } else {
        constexpr int LPB = 16 / V;
        amax = block_amax<LPB>(amax);
        const bool special = !(amax <= 3.402823466e38f);     // NaN or Inf in the block
        const uint8_t sc = special ? (uint8_t)0x7F : e4m3_of(amax * p.q_inv6s);
        const float sv = special ? 0.f : e4m3_value(sc);
        uint32_t packed = 0u;
        if (sv > 0.f) {
            // fast reciprocal (CUDA documents <= 2 ulp): the code decision
            // tolerance covers it (a few 1e-7 against 2.5e-6)
            const float rcp = __fdividef(1.f, sv * p.q_scale);
#pragma unroll
            for (int k = 0; k < V / 2; ++k) packed |= e2m1x2(a[2 * k] * rcp, a[2 * k + 1] * rcp) << (8 * k);
        }
        if (valid) {
            char *dst = static_cast<char *>(p.y) + row * (p.row_elems / 2) + (int64_t)u * (V / 2);
            if constexpr (V == 8) {
                asm volatile("st.global.u32 [%0], %1;" : : "l"(dst), "r"(packed) : "memory");
            } else {
                asm volatile("st.global.u16 [%0], %1;" : : "l"(dst), "h"((unsigned short)packed) : "memory");
            }
            if (t % LPB == 0) static_cast<uint8_t *>(p.scales)[row * (p.row_elems / 16) + u / LPB] = sc;
        }
    }
}

// The register kernel's body: blocks stride over row groups of RPB rows.
template <typename T, int GT, int CH, bool RES, int WM, bool HEADS, int OUT>
__device__ __forceinline__ void rms_reg_rows(const Params &p) {
    constexpr bool W = WM != kNoWeight;
    constexpr bool W_DIRECT = W && GT <= 32 && OUT == kOutT;   // per-lane weight loads (below)
    static_assert(!(HEADS && RES), "head rows take no residual");
    static_assert(OUT == kOutT || (!HEADS && GT >= 32 / T::kVec), "block-scaled output: contiguous rows, "
                                                                  "a block's lanes in one row group");
    constexpr int V = T::kVec;
    constexpr int BLOCK = reg_block_threads(GT);
    constexpr int RPB = BLOCK / GT;               // row groups a block can hold
    constexpr int LANES = GT < 32 ? GT : 32;      // butterfly width
    constexpr int WPR = GT > 32 ? GT / 32 : 1;    // warps per row
    static_assert((GT & (GT - 1)) == 0 && GT >= 4 && GT <= 1024, "GT: power of two in [4, 1024]");
    __shared__ float red[2][RPB][WPR];

    const int tid = threadIdx.x;
    const int slot = tid / GT;
    const int t = tid % GT;
    const int nch = p.units;

    // before the wait: the block's first row group into L2 (contiguous rows,
    // whose row group is one contiguous range)
    if constexpr (!HEADS) {
        const int n = RPB == 1 ? 1 : (p.rpb >= 1 && p.rpb <= RPB ? p.rpb : RPB);
        if (tid == 0) prefetch_rows_l2<RES>(p.x, p.res, p.row_bytes, p.rows, (int64_t)blockIdx.x * n, n);
    }
    pdl_wait_for_inputs();
    pdl_allow_dependents();

    // w (and w2 for head rows) is the same for every row.  Rows of a warp or
    // less (W_DIRECT) load their weight chunks per lane right after their x
    // chunks: no block barrier, and L1 serves the block's other rows
    // (measured on GB300: bf16 4096 x 576 3.07 -> 3.01 us, Q+K heads of 8192
    // tokens 26.5 -> 25.4 us).  Otherwise w is staged once per block in
    // shared memory (dynamic, units * 16 bytes per weight; the host sizes it
    // for every REG plan with a weight) after the first row's loads are
    // issued, so the two memory round trips overlap.
    extern __shared__ Chunk w_smem[];
    bool w_staged = false;

    int parity = 0;
    // p.rpb (1 .. RPB) rows a block iteration: RPB, or one row a block when a
    // launch has no more rows than the device has SMs (each row then gets an
    // SM of its own; the idle row slots load and store nothing).  Which block
    // takes a row changes no result.
    // the host passes 1..RPB; a block of one row slot needs no run-time count
    const int rpb = RPB == 1 ? 1 : (p.rpb >= 1 && p.rpb <= RPB ? p.rpb : RPB);
    const int64_t step = (int64_t)gridDim.x * rpb;
    for (int64_t first = (int64_t)blockIdx.x * rpb; first < p.rows; first += step) {
        const int64_t row = first + slot;
        const bool row_ok = (RPB == 1 || slot < rpb) && row < p.rows;
        int64_t off = 0, yoff = 0;
        int wsel = 0;
        if (row_ok) row_offsets<HEADS>(p, row, off, yoff, wsel);

        // A1: load the row's chunks (zeros where a slot is past the row end)
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
        Chunk wc[W_DIRECT ? CH : 1];
        if constexpr (W_DIRECT) {
            const char *wp = static_cast<const char *>(wsel ? p.w2 : p.w);
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int u = c * GT + t;
                if (row_ok && u < nch)
                    wc[c] = ld_readonly16(wp + (int64_t)u * 16);
                else
                    wc[c] = Chunk{{0u, 0u, 0u, 0u}};
            }
        }
        if constexpr (W && !W_DIRECT) {
            if (!w_staged) {   // first iteration of the block (uniform across it)
                for (int i = tid; i < nch; i += BLOCK)
                    w_smem[i] = ld_readonly16(static_cast<const char *>(p.w) + (int64_t)i * 16);
                if constexpr (HEADS) {
                    for (int i = tid; i < nch; i += BLOCK)
                        w_smem[nch + i] = ld_readonly16(static_cast<const char *>(p.w2) + (int64_t)i * 16);
                }
                __syncthreads();
                w_staged = true;
            }
        }
        // A2: h = RN_T(x + residual), written out as residual_out
        if constexpr (RES) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int u = c * GT + t;
                float a[V], b[V];
                unpack(hc[c], a, T{});
                unpack(rc[c], b, T{});
#pragma unroll
                for (int e = 0; e < V; ++e) a[e] = add_round(a[e], b[e], T{});
                hc[c] = pack(a, T{});
                if (row_ok && u < nch)
                    st16(static_cast<char *>(p.res_out) + yoff + (int64_t)u * 16, hc[c]);
            }
        }
        // A3: squares into V accumulators, chunk order; zero slots add +0 exactly
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            float a[V];
            unpack(hc[c], a, T{});
            sq_accumulate(a, acc);
        }
        float sum = tree_sum(acc);
        // A4: butterfly across the row's lanes of this warp
        sum = butterfly_sum<LANES>(sum);
        // A5: fixed-order combine across the row's warps
        if constexpr (WPR > 1) {
            if ((tid & 31) == 0) red[parity][slot][t / 32] = sum;
            __syncthreads();
            float v[WPR];
#pragma unroll
            for (int i = 0; i < WPR; ++i) v[i] = red[parity][slot][i];
            sum = tree_sum(v);
            parity ^= 1;   // the next iteration writes the other buffer
        }
        // A6: the row's scale
        const float r = rsqrtf(sum / p.hidden_f + p.eps);
        // A7, block-scaled forms: values, block scale, codes
        if constexpr (OUT != kOutT) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int u = c * GT + t;
                const bool valid = row_ok && u < nch;     // uniform over a block's lanes
                float a[V];
                unpack(hc[c], a, T{});
                float wv[V];
                if constexpr (W) {
                    unpack(w_smem[valid ? u : 0], wv, T{});
                } else {
#pragma unroll
                    for (int e = 0; e < V; ++e) wv[e] = 1.f;
                }
                scale_out_pairs<WM>(a, r, wv, p.w_bias);
                store_quantised<V, OUT>(a, valid, p, row, u, t);
            }
            continue;
        }
        // A7: y = RN_T(h * r * w)   (or h * r, or h * r * (w + bias))
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int u = c * GT + t;
            if (row_ok && u < nch) {
                float a[V];
                unpack(hc[c], a, T{});
                float wv[V];
                if constexpr (W_DIRECT) {
                    unpack(wc[c], wv, T{});
                } else if constexpr (W) {
                    unpack(w_smem[wsel * nch + u], wv, T{});
                } else {
#pragma unroll
                    for (int e = 0; e < V; ++e) wv[e] = 1.f;
                }
                scale_out_pairs<WM>(a, r, wv, p.w_bias);
                st16(static_cast<char *>(p.y) + yoff + (int64_t)u * 16, pack(a, T{}));
            }
        }
    }
}

// Plain output: the launch bound names the block size only.
template <typename T, int GT, int CH, bool RES, int WM, bool HEADS>
__global__ void __launch_bounds__(reg_block_threads(GT)) rms_reg_kernel(const Params p) {
    rms_reg_rows<T, GT, CH, RES, WM, HEADS, kOutT>(p);
}

// Resident blocks the block-scaled epilogues are budgeted for: four 256-thread
// blocks (64 registers a thread) up to 4 chunks, where they fit without
// spilling more than a word; measured on GB300, four blocks beat the three
// that the unbudgeted 76 registers allow (MXFP8 16384 x 2048 with residual
// 0.940 -> 0.965 of peak, NVFP4 65536 x 8192 0.954 -> 1.004).  8 chunks would
// spill.
__host__ __device__ constexpr int quant_min_blocks(int gt, int ch) {
    return (reg_block_threads(gt) == 256 && ch <= 4) ? 4 : 1;
}

// MXFP8 / NVFP4 output (contiguous rows).
template <typename T, int GT, int CH, bool RES, int WM, int OUT>
__global__ void __launch_bounds__(reg_block_threads(GT), quant_min_blocks(GT, CH)) rms_quant_kernel(const Params p) {
    rms_reg_rows<T, GT, CH, RES, WM, false, OUT>(p);
}

// ------------------------------------------------------- two-pass kernel
// Units are VE elements: VE == T::kVec (one 16-byte chunk) or 1 (a scalar).
// Raw units stay packed in registers until they are used.

template <typename T, int VE>
struct UnitIO;

template <typename T>
struct UnitIO<T, T::kVec> {
    static constexpr int VE = T::kVec;
    using Raw = Chunk;
    __device__ static Raw zero() { return Chunk{{0u, 0u, 0u, 0u}}; }
    __device__ static Raw load_first(const void *base, int64_t u) {
        return ld_keep_l2_16(static_cast<const char *>(base) + u * 16);
    }
    __device__ static Raw load_last(const void *base, int64_t u) {
        return ld_stream16(static_cast<const char *>(base) + u * 16);
    }
    __device__ static Raw load_w(const void *base, int64_t u) {
        return ld_readonly16(static_cast<const char *>(base) + u * 16);
    }
    __device__ static void widen(const Raw &r, float (&f)[VE]) { unpack(r, f, T{}); }
    __device__ static void store(void *base, int64_t u, const float (&f)[VE]) {
        st16(static_cast<char *>(base) + u * 16, pack(f, T{}));
    }
};

// Scalar units: the raw value is the element's bit pattern in 32 bits.
__device__ __forceinline__ uint32_t ld_bits(const void *p, int64_t i, BF16, int hint) {
    unsigned short v;
    const void *a = static_cast<const uint16_t *>(p) + i;
    if (hint == 0)
        asm volatile("ld.global.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(a));
    else if (hint == 1)
        asm volatile("ld.global.cs.u16 %0, [%1];" : "=h"(v) : "l"(a));
    else
        asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(a));
    return (uint32_t)v;
}
__device__ __forceinline__ uint32_t ld_bits(const void *p, int64_t i, F32, int hint) {
    uint32_t v;
    const void *a = static_cast<const float *>(p) + i;
    if (hint == 0)
        asm volatile("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(a));
    else if (hint == 1)
        asm volatile("ld.global.cs.u32 %0, [%1];" : "=r"(v) : "l"(a));
    else
        asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(a));
    return v;
}
__device__ __forceinline__ float widen_bits(uint32_t b, BF16) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float widen_bits(uint32_t b, F32) { return __uint_as_float(b); }
__device__ __forceinline__ void st_scalar(void *p, int64_t i, float v, BF16) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    unsigned short s = *reinterpret_cast<unsigned short *>(&b);
    asm volatile("st.global.u16 [%0], %1;" : : "l"(static_cast<uint16_t *>(p) + i), "h"(s) : "memory");
}
__device__ __forceinline__ void st_scalar(void *p, int64_t i, float v, F32) {
    asm volatile("st.global.f32 [%0], %1;" : : "l"(static_cast<float *>(p) + i), "f"(v) : "memory");
}

template <typename T>
struct UnitIO<T, 1> {
    static constexpr int VE = 1;
    using Raw = uint32_t;
    __device__ static Raw zero() { return 0u; }
    __device__ static Raw load_first(const void *base, int64_t u) { return ld_bits(base, u, T{}, 0); }
    __device__ static Raw load_last(const void *base, int64_t u) { return ld_bits(base, u, T{}, 1); }
    __device__ static Raw load_w(const void *base, int64_t u) { return ld_bits(base, u, T{}, 2); }
    __device__ static void widen(const Raw &r, float (&f)[1]) { f[0] = widen_bits(r, T{}); }
    __device__ static void store(void *base, int64_t u, const float (&f)[1]) {
        st_scalar(base, u, f[0], T{});
    }
};

template <typename T, int VE, int BLOCK, bool RES, int WM, bool HEADS>
__global__ void __launch_bounds__(BLOCK, 1)
rms_loop_kernel(const Params p) {
    constexpr bool W = WM != kNoWeight;
    static_assert(!(HEADS && RES), "head rows take no residual");
    using IO = UnitIO<T, VE>;
    using Raw = typename IO::Raw;
    constexpr int NACC = 8;                          // per-thread accumulators
    // units in flight per step: without a residual the first pass has no
    // second input, so it takes twice the units to keep as many bytes in
    // flight (an accumulator's sequence of units is the same for any U)
    constexpr int U = VE == 1 ? NACC : (RES ? 2 : 4);
    constexpr int NW = BLOCK / 32;
    static_assert(BLOCK % 32 == 0 && (NW & (NW - 1)) == 0, "BLOCK: power-of-two warps");
    static_assert((U * VE) % NACC == 0 || NACC % (U * VE) == 0, "accumulator cycle");
    __shared__ float red[2][NW];

    const int tid = threadIdx.x;
    const int64_t nunits = p.units;
    int parity = 0;
    pdl_wait_for_inputs();
    pdl_allow_dependents();

    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        int64_t off, yoff;
        int wsel;
        row_offsets<HEADS>(p, row, off, yoff, wsel);
        const void *xr = static_cast<const char *>(p.x) + off;
        const void *rr = RES ? static_cast<const char *>(p.res) + off : nullptr;
        void *hr = RES ? static_cast<char *>(p.res_out) + yoff : nullptr;
        void *yr = static_cast<char *>(p.y) + yoff;
        const void *wr = wsel ? p.w2 : p.w;

        // pass 1: h (and residual_out), sum of squares.  Element e of the
        // j-th unit of a step feeds accumulator (j * VE + e) % NACC.
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
                    float b[VE];
                    IO::widen(rb[j], b);
#pragma unroll
                    for (int e = 0; e < VE; ++e) a[e] = add_round(a[e], b[e], T{});
                    if (u < nunits) IO::store(hr, u, a);
                }
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                    const int k = (j * VE + e) % NACC;
                    acc[k] = fmaf(a[e], a[e], acc[k]);
                }
            }
        }
        float sum = tree_sum(acc);
        sum = butterfly_sum<32>(sum);
        if constexpr (NW > 1) {
            if ((tid & 31) == 0) red[parity][tid / 32] = sum;
            __syncthreads();
            float v[NW];
#pragma unroll
            for (int i = 0; i < NW; ++i) v[i] = red[parity][i];
            sum = tree_sum(v);
            parity ^= 1;
        }
        const float r = rsqrtf(sum / p.hidden_f + p.eps);

        // pass 2: re-read h (x, or residual_out written above by this same
        // thread) and write y
        const void *src = RES ? static_cast<const void *>(hr) : xr;
        for (int64_t base = tid; base < nunits; base += (int64_t)BLOCK * U) {
            Raw ha[U];
            Raw wa[W ? U : 1];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t u = base + (int64_t)j * BLOCK;
                ha[j] = u < nunits ? IO::load_last(src, u) : IO::zero();
                if constexpr (W) wa[j] = u < nunits ? IO::load_w(wr, u) : IO::zero();
            }
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t u = base + (int64_t)j * BLOCK;
                float a[VE];
                IO::widen(ha[j], a);
                float wv[VE];
                if constexpr (W) {
                    IO::widen(wa[j], wv);
                } else {
#pragma unroll
                    for (int e = 0; e < VE; ++e) wv[e] = 1.f;
                }
#pragma unroll
                for (int e = 0; e < VE; ++e) a[e] = scale_out<WM>(a[e], r, wv[e], p.w_bias);
                if (u < nunits) IO::store(yr, u, a);
            }
        }
    }
}

}  // namespace rrn
