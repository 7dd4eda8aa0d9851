// rmsnorm_cluster.cuh -- the fused RMSNorm of rows too long for one block's
// registers, split over the blocks of a thread-block cluster.
//
// The op per row is the one of rmsnorm_kernels.cuh: h = RN_T(x + residual)
// (stored as residual_out), y = RN_T(h * rsqrt(mean(h^2) + eps) * w);
// definition: "Building a GPU compiler from scratch (Emmy)", section "Tensor
// IR".  Its section "Loop IR" keeps the row's statistic on chip and reads
// every byte once; for a row past what one block holds in registers, the
// blocks of a cluster hold it together here, which keeps that single pass:
//
//  * A cluster of C blocks (2..8, the portable cluster size) owns a row; block
//    q of the cluster owns the slice of units [q*S, (q+1)*S), S = 256 * CH
//    16-byte units (16 KB with CH = 4, 20 KB with CH = 5, 32 KB with CH = 8),
//    thread t the units
//    q*S + c*256 + t, so a warp's loads of one chunk slot are 512 contiguous
//    bytes.  The slice lives in registers from its load to its store.
//  * Each block reduces its slice exactly as the register kernel's CTA regime
//    does (chunk-order accumulators, a fixed tree over them, xor butterflies,
//    a fixed tree over the 8 warps), then writes its partial sum into every
//    block of the cluster (distributed shared memory: mapa +
//    st.shared::cluster), and one cluster barrier (arrive.release /
//    wait.acquire) makes all C partials visible in each block.  Every block
//    then sums the 8 partial slots in a fixed tree, the slots of absent
//    blocks (and of blocks past the row end) holding +0.
//  * So a row's result depends on its length, dtype and CH alone -- not on
//    the cluster size, the grid or the row count -- and no atomics are used.
//  * The wait is the hardware cluster barrier: every thread of every block of
//    a cluster reaches it once per row (uniform control flow: the row loop's
//    bounds are the same for all blocks of a cluster), and no block touches
//    another's shared memory after the barrier, so a block may exit as soon
//    as its row is done.  No spin-wait is involved.
//  * Before waiting on the kernel ahead of it (programmatic dependent launch)
//    a block asks for its slice of its first row to be prefetched into L2.
//
// Measured on GB300 (bf16 rows with a residual and a weight, against the
// kernels these rows ran on before): 48 KB rows 0.936 -> 0.982 of the
// measured HBM peak, 64 KB 0.946 -> 0.986, 80 KB 0.949 -> 0.964 with five
// 16 KB slices, 0.976 with four 20 KB slices (all against the bulk-copy
// kernel), 128 KB 0.915 -> 0.959 (against the two-pass
// kernel); fp32 rows of 160 KB 0.969 -> 1.025 and of 256 KB 0.934 -> 1.006
// with 32 KB slices.  Without a residual a block moves half the bytes per
// barrier and the bulk-copy kernel stays faster (64 KB rows 0.709 against
// 1.029), so only rows with a residual are planned here.
#pragma once

#include "kernel_table.h"
#include "rmsnorm_kernels.cuh"

namespace rrn {

// Resident blocks each slice size is compiled for: four (64 registers a
// thread) for 16 and 20 KB slices, three (85) for 32 KB slices; measured on
// GB300, fp32 rows of 256 KB with 32 KB slices 1.006 of peak at three
// blocks, 0.907 at two; bf16 rows of 80 KB with 20 KB slices 0.976 at four
// blocks, 0.956 at three.
__host__ __device__ constexpr int cluster_min_blocks(int ch) { return ch <= 5 ? 4 : 3; }

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_ctas() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// v into the shared-memory word that `local` names, in block `rank` of the
// cluster (its own shared memory when rank is the caller's).
__device__ __forceinline__ void st_cluster_f32(const float *local, uint32_t rank, float v) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" : : "r"(ra), "f"(v) : "memory");
}

// Every thread of every block of the cluster: the stores before it are
// visible to every block after it.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;" : : : "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" : : : "memory");
}

// The slice [u0, u0 + S) of row `row` (contiguous rows) into L2, by thread 0.
template <bool RES, int S>
__device__ __forceinline__ void prefetch_slice_l2(const Params &p, int64_t row, int u0) {
    const int64_t b0 = (int64_t)u0 * 16;
    if (row >= p.rows || b0 >= p.row_bytes) return;
    const int64_t rest = p.row_bytes - b0;
    const unsigned n = (unsigned)(rest < (int64_t)S * 16 ? rest : (int64_t)S * 16);
    prefetch_l2(static_cast<const char *>(p.x) + row * p.x_stride + b0, n);
    if constexpr (RES) prefetch_l2(static_cast<const char *>(p.res) + row * p.x_stride + b0, n);
}

template <typename T, int CH, bool RES, int WM>
__global__ void __launch_bounds__(kClusterGT, cluster_min_blocks(CH)) rms_cluster_kernel(const Params p) {
    constexpr bool W = WM != kNoWeight;
    constexpr int V = T::kVec;
    constexpr int GT = kClusterGT;
    constexpr int NW = GT / 32;
    constexpr int S = GT * CH;   // 16-byte units of a block's slice
    __shared__ float red[2][NW];
    __shared__ float part[2][kClusterMaxCtas];

    const int tid = threadIdx.x;
    const uint32_t q = cluster_rank();
    const uint32_t ncta = cluster_ctas();
    if (ncta > (uint32_t)kClusterMaxCtas) return;   // the host never launches it (uniform over a cluster)
    const int64_t first = cluster_index();
    const int64_t step = cluster_count();
    const int nch = p.units;
    const int u0 = (int)q * S;

    if (tid == 0) prefetch_slice_l2<RES, S>(p, first, u0);
    pdl_wait_for_inputs();
    pdl_allow_dependents();

    // The partial-sum buffers alternate between rows: a block that moves on
    // writes the next row's partials into the other buffer, and it can only
    // come back to this one after every block of the cluster has passed the
    // next row's barrier, i.e. has read this row's partials.
    int parity = 0;
    for (int64_t row = first; row < p.rows; row += step) {
        const int64_t off = row * p.x_stride, yoff = row * p.y_stride;
        // A1: the slice's chunks (zeros past the row end)
        Chunk hc[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int u = u0 + c * GT + tid;
            hc[c] = u < nch ? ld_stream16(static_cast<const char *>(p.x) + off + (int64_t)u * 16)
                            : Chunk{{0u, 0u, 0u, 0u}};
        }
        // A2: h = RN_T(x + residual), written out as residual_out
        if constexpr (RES) {
            Chunk rc[CH];
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int u = u0 + c * GT + tid;
                rc[c] = u < nch ? ld_stream16(static_cast<const char *>(p.res) + off + (int64_t)u * 16)
                                : Chunk{{0u, 0u, 0u, 0u}};
            }
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int u = u0 + c * GT + tid;
                float a[V], b[V];
                unpack(hc[c], a, T{});
                unpack(rc[c], b, T{});
#pragma unroll
                for (int e = 0; e < V; ++e) a[e] = add_round(a[e], b[e], T{});
                hc[c] = pack(a, T{});
                if (u < nch) st16(static_cast<char *>(p.res_out) + yoff + (int64_t)u * 16, hc[c]);
            }
        }
        // the weight's slice, issued once the residual's registers are free;
        // it lands while the row is reduced
        Chunk wc[W ? CH : 1];
        if constexpr (W) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int u = u0 + c * GT + tid;
                wc[c] = u < nch ? ld_readonly16(static_cast<const char *>(p.w) + (int64_t)u * 16)
                                : Chunk{{0u, 0u, 0u, 0u}};
            }
        }
        // A3: squares into V accumulators, chunk order
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
        // A4, A5: the warp's lanes, then the block's 8 warps
        sum = butterfly_sum<32>(sum);
        if ((tid & 31) == 0) red[parity][tid / 32] = sum;
        __syncthreads();
        {
            float v[NW];
#pragma unroll
            for (int i = 0; i < NW; ++i) v[i] = red[parity][i];
            sum = tree_sum(v);
        }
        // the block's partial into slot q of every block of the cluster
        if (tid < (int)ncta) st_cluster_f32(&part[parity][q], (uint32_t)tid, sum);
        cluster_barrier();
        {
            float v[kClusterMaxCtas];
#pragma unroll
            for (int i = 0; i < kClusterMaxCtas; ++i) v[i] = i < (int)ncta ? part[parity][i] : 0.f;
            sum = tree_sum(v);
        }
        parity ^= 1;
        // A6: the row's scale
        const float r = rsqrtf(sum / p.hidden_f + p.eps);
        // A7: y = RN_T(h * r * w)   (or h * r, or h * r * (w + bias), or the cast order)
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int u = u0 + c * GT + tid;
            if (u < nch) {
                float a[V];
                unpack(hc[c], a, T{});
                float wv[V];
                if constexpr (W) {
                    unpack(wc[c], wv, T{});
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

}  // namespace rrn
