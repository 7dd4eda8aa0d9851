// rmsnorm_tma.cuh -- RMSNorm with the row staged in shared memory by bulk
// (TMA) copies: the kernel for long rows (planned past 32 KB, where it beats
// holding 512 x 8 chunks in registers) and for block-scaled outputs of rows
// too long for registers.  "CuTeDSL at Perplexity", section "QK Norm": rows
// of thousands of elements reduce through shared memory as well as
// registers; "Building a GPU compiler from scratch ... (Emmy)", schedule
// codec: TMA copies guarded by barriers, double buffered.
//
// The op and the per-thread arithmetic are those of the register kernel with
// 512 threads a row (chunk u of a row belongs to thread u mod 512, the
// thread adds its squares in increasing u, then the warp butterfly and the
// fixed-order tree over the 16 warps), so for a row that both kernels can
// take the two give the same bits.  What differs is where the row waits
// between the reduction and the scaling: in a ring of shared-memory pieces
// instead of registers.
//
// Block: 16 consumer warps (512 threads) and three producer warps.  A row is
// cut into pieces of 512 x 16 x PC bytes (the last one shorter); piece k holds
// the chunks c = k*PC .. k*PC + PC - 1 of every consumer thread.  Up to three
// rings of pieces share the block's shared memory: x, the residual and the
// weight.  The weight ring, when there is one, holds the whole weight (one
// slot a piece, copied once per block and never released); when the slots
// are better spent on x (long rows: the x ring then keeps fewer than two
// spare slots beside a resident weight), there is no weight ring and the
// consumers read the weight's chunks straight from global memory, where
// every block after the first finds them in L2 (measured on GB300, bf16
// 2048 x 65536 without a residual 0.92 -> 0.96 of the measured peak against
// a weight streamed through a ring, 2730 x 49152 0.93 -> 0.97 against a
// resident weight with one spare x slot; with two or more spare slots the
// resident weight is faster: 4096 x 32768 1.03 against 0.90).
// Each slot has a "full" mbarrier (the producer's arrival plus the copy's
// byte count) and an "empty" mbarrier (one arrival per consumer warp).  One
// lane of each producer warp walks the block's rows (blockIdx.x, + gridDim.x,
// ...) and their pieces in order, waits until its ring's next slot is empty,
// and issues one cp.async.bulk global -> shared copy of the piece that
// completes on the slot's full barrier.  The consumers take the same walk:
// pass 1 waits for each x piece (and residual piece), adds the residual (the
// sum is written back into the x piece and out as residual_out), accumulates
// the squares and releases the residual slot; after the row's reduction,
// pass 2 waits for each weight piece (when the weight has a ring), scales,
// writes y and releases the x slot (and a streamed weight slot).  As long as
// the x ring has a slot for
// every piece of a row, no producer is ever blocked by the row being
// reduced, and the next rows stream in while this row is scaled.  Both passes
// read x and the residual from shared memory only, so no warp waits on an HBM
// round trip (the weight, when it is not resident, comes from L2).
//
// Every wait is bounded (Params::wait_ns on the globaltimer, one second in
// every library launch).  A wait that runs out marks the thread failed; a
// failed thread skips its later waits but keeps the same control flow (so
// every barrier is still reached), and a warp whose lane 0 has failed releases
// no slot from then on.  A slot is released, that is, only by warps that saw
// its copy land, so a producer never starts a copy into a slot whose previous
// copy may still be in flight (which would arrive on the slot's "full"
// barrier before its phase completed); a producer that waits for such a slot
// gives up in turn.  The block counts itself in g_tma_timeouts, and before it
// exits one thread waits (bounded again) for every copy still in flight into
// its shared memory.
//
// This header defines the counter below, so one translation unit (tma.cu)
// includes it.
#pragma once

#include "kernel_table.h"
#include "rmsnorm_kernels.cuh"

namespace rrn {

constexpr int kTmaWarps = kTmaGT / 32;          // consumer warps

// Blocks that gave up on a wait since the library was loaded.
__device__ unsigned int g_tma_timeouts = 0;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" : : "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" : : "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 : : "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the completion of the barrier phase of the given parity; false if
// limit_ns nanoseconds passed first.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Bulk copy global -> shared of `bytes` bytes (a multiple of 16; both
// addresses 16-byte aligned), completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 : : "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ Chunk lds16(const void *p) {
    Chunk c;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(c.u[0]), "=r"(c.u[1]), "=r"(c.u[2]), "=r"(c.u[3])
                 : "r"(smem_u32(p)));
    return c;
}

__device__ __forceinline__ void sts16(void *p, const Chunk &c) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                 : : "r"(smem_u32(p)), "r"(c.u[0]), "r"(c.u[1]), "r"(c.u[2]), "r"(c.u[3])
                 : "memory");
}

// Barrier over the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" : : "n"(kTmaGT) : "memory");
}

// The slots of one ring: barriers and memory.  Slot s holds a piece at
// mem + s * piece bytes; full[s] completes when the piece has landed,
// empty[s] when every consumer warp has released it.
struct Ring {
    uint64_t *full;
    uint64_t *empty;
    unsigned char *mem;
    unsigned n;
};

// Producer walk (one lane): piece k of each of the block's rows in order --
// or, with `once`, the pieces of a single row-sized source -- each into the
// ring's next slot once that slot is empty.  `issued` receives the number of
// copies issued; false if a wait for an empty slot ran out.
template <int PIECE>
__device__ __forceinline__ bool feed_ring(const Ring &R, const char *src, int64_t row_stride, const Params &p,
                                          int pieces, int64_t row_bytes, bool once, unsigned &issued) {
    unsigned q = 0;
    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const char *base = src + (once ? 0 : row * row_stride);
        for (int k = 0; k < pieces; ++k) {
            const unsigned s = q % R.n, n = q / R.n;
            if (n > 0 && !mbar_wait_bounded(&R.empty[s], (n - 1) & 1u, p.wait_ns)) {
                issued = q;
                return false;
            }
            const int64_t off = (int64_t)k * PIECE;
            const unsigned bytes = (unsigned)(row_bytes - off < PIECE ? row_bytes - off : PIECE);
            mbar_arrive_expect_tx(&R.full[s], bytes);
            bulk_g2s(R.mem + (size_t)s * PIECE, base + off, bytes, &R.full[s]);
            ++q;
        }
        if (once) break;
    }
    issued = q;
    return true;
}

// Waits (bounded) for the last copy issued into each slot of a ring.
__device__ __forceinline__ void drain_ring(const Ring &R, unsigned issued, unsigned long long limit_ns) {
    for (unsigned j = issued > R.n ? issued - R.n : 0u; j < issued; ++j)
        (void)mbar_wait_bounded(&R.full[j % R.n], (j / R.n) & 1u, limit_ns);
}

// sx, sr, sw: slots of the x, residual and weight rings (sr = 0 without a
// residual, sw = 0 without a weight ring).  sx >= pieces; sw >= pieces makes
// the weight resident (copied once per block, never released); fewer weight
// slots stream it.  WG: there is no weight ring, the consumers read the
// weight from global memory (the library plans resident weights and WG; the
// streaming form is kept for any other split a caller might pass).
// OUT: kOutT writes y in the I/O type; kOutMxfp8 / kOutNvfp4 write the
// block-scaled codes and scales (the register kernel's epilogue, with the
// same lane layout: a block's chunks sit in consecutive threads of a piece).
template <typename T, bool RES, int WM, int PC, int OUT = kOutT, bool WG = false>
__global__ void __launch_bounds__(kTmaBlock, 1)
rms_tma_kernel(const Params p, const int sx, const int sr, const int sw) {
    constexpr bool W = WM != kNoWeight;
    constexpr bool WR = W && !WG;   // the weight comes through a ring
    constexpr int V = T::kVec;
    constexpr int GT = kTmaGT;
    constexpr int PIECE = kTmaGT * 16 * PC;   // tma_piece_bytes(PC)
    __shared__ float red[2][kTmaWarps];
    __shared__ int s_failed;
    __shared__ unsigned s_issued[3];
    extern __shared__ __align__(128) unsigned char tma_smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(tma_smem);
    uint64_t *empty = full + kTmaMaxSlots;
    unsigned char *mem = tma_smem + kTmaBarBytes;
    const Ring X{full, empty, mem, (unsigned)sx};
    const Ring Rr{full + sx, empty + sx, mem + (size_t)sx * PIECE, (unsigned)(sr > 0 ? sr : 1)};
    const Ring Wr{full + sx + sr, empty + sx + sr, mem + (size_t)(sx + sr) * PIECE, (unsigned)(sw > 0 ? sw : 1)};

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int nch = p.units;
    const int64_t row_bytes = p.row_bytes;
    const int pieces = (int)((row_bytes + PIECE - 1) / PIECE);
    const bool w_resident = sw >= pieces;
    if constexpr (WR) {
        // a weight ring needs a slot: without one, count the launch as failed
        // and touch nothing (every thread leaves here, before any barrier)
        if (sw < 1) {
            if (threadIdx.x == 0) atomicAdd(&g_tma_timeouts, 1u);
            return;
        }
    }

    if (tid == 0) {
        for (int s = 0; s < sx + sr + sw; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kTmaWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        s_failed = 0;
        s_issued[0] = s_issued[1] = s_issued[2] = 0;
    }
    __syncthreads();
    // before the wait: the block's first row into L2 (see prefetch_rows_l2)
    if (tid == 0) prefetch_rows_l2<RES>(p.x, p.res, row_bytes, p.rows, (int64_t)blockIdx.x, 1);
    pdl_wait_for_inputs();
    pdl_allow_dependents();

    if (warp >= kTmaWarps) {
        // ------------------------------------------ producers: x, residual, w
        const int role = warp - kTmaWarps;
        if (lane == 0) {
            unsigned issued = 0;
            bool ok = true;
            if (role == 0)
                ok = feed_ring<PIECE>(X, static_cast<const char *>(p.x), row_bytes, p, pieces, row_bytes, false,
                                      issued);
            else if (role == 1 && RES)
                ok = feed_ring<PIECE>(Rr, static_cast<const char *>(p.res), row_bytes, p, pieces, row_bytes, false,
                                      issued);
            else if (role == 2 && WR)
                ok = feed_ring<PIECE>(Wr, static_cast<const char *>(p.w), 0, p, pieces, row_bytes, w_resident,
                                      issued);
            s_issued[role] = issued;
            if (!ok) s_failed = 1;
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- consumers
        const int t = tid;
        unsigned qx = 0, qr = 0, qw = 0;
        bool ok = true;
        int par = 0;
        for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
            const int64_t roff = row * row_bytes;
            float acc[V];
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = 0.f;

            // pass 1: A1-A3 over the pieces as they land
            for (int k = 0; k < pieces; ++k) {
                const unsigned xs = (qx + (unsigned)k) % X.n;
                if (ok) ok = mbar_wait_bounded(&X.full[xs], ((qx + (unsigned)k) / X.n) & 1u, p.wait_ns);
                unsigned char *xp = X.mem + (size_t)xs * PIECE;
                unsigned rs = 0;
                const unsigned char *rp = nullptr;
                if constexpr (RES) {
                    rs = qr % Rr.n;
                    if (ok) ok = mbar_wait_bounded(&Rr.full[rs], (qr / Rr.n) & 1u, p.wait_ns);
                    rp = Rr.mem + (size_t)rs * PIECE;
                }
                // every shared-memory load of the piece is issued before the
                // first is used, so a warp keeps PC (2 PC) of them in flight
                Chunk xa[PC], ra[RES ? PC : 1];
#pragma unroll
                for (int j = 0; j < PC; ++j) {
                    const int so = (j * GT + t) * 16;
                    if ((k * PC + j) * GT + t < nch) {
                        xa[j] = lds16(xp + so);
                        if constexpr (RES) ra[j] = lds16(rp + so);
                    }
                }
#pragma unroll
                for (int j = 0; j < PC; ++j) {
                    const int u = (k * PC + j) * GT + t;
                    if (u < nch) {
                        const int so = (j * GT + t) * 16;
                        float a[V];
                        unpack(xa[j], a, T{});
                        if constexpr (RES) {
                            float b[V];
                            unpack(ra[j], b, T{});
#pragma unroll
                            for (int e = 0; e < V; ++e) a[e] = add_round(a[e], b[e], T{});
                            const Chunk h = pack(a, T{});
                            sts16(xp + so, h);
                            st16(static_cast<char *>(p.res_out) + roff + (int64_t)u * 16, h);
                        }
                        sq_accumulate(a, acc);
                    }
                }
                if constexpr (RES) {   // the residual piece is used up
                    __syncwarp();
                    if (lane == 0 && ok) mbar_arrive(&Rr.empty[rs]);
                    ++qr;
                }
            }
            // A4-A6: butterfly, fixed-order tree over the 16 warps, the scale
            float sum = tree_sum(acc);
            sum = butterfly_sum<32>(sum);
            if (lane == 0) red[par][warp] = sum;
            consumer_sync();
            float v[kTmaWarps];
#pragma unroll
            for (int i = 0; i < kTmaWarps; ++i) v[i] = red[par][i];
            sum = tree_sum(v);
            par ^= 1;
            const float r = rsqrtf(sum / p.hidden_f + p.eps);

            // pass 2: A7 per piece, then release the x (and w) slots
            for (int k = 0; k < pieces; ++k) {
                const unsigned xs = (qx + (unsigned)k) % X.n;
                unsigned char *xp = X.mem + (size_t)xs * PIECE;
                unsigned ws = 0;
                const unsigned char *wp = nullptr;
                if constexpr (WR) {
                    ws = w_resident ? (unsigned)k : qw % Wr.n;
                    const unsigned wpar = w_resident ? 0u : (qw / Wr.n) & 1u;
                    if (ok) ok = mbar_wait_bounded(&Wr.full[ws], wpar, p.wait_ns);
                    wp = Wr.mem + (size_t)ws * PIECE;
                }
                Chunk xa[OUT == kOutT ? PC : 1], wa[OUT == kOutT && W ? PC : 1];
                if constexpr (OUT == kOutT) {   // loads first, as in pass 1
#pragma unroll
                    for (int j = 0; j < PC; ++j) {
                        const int so = (j * GT + t) * 16;
                        if ((k * PC + j) * GT + t < nch) {
                            xa[j] = lds16(xp + so);
                            if constexpr (WR)
                                wa[j] = lds16(wp + so);
                            else if constexpr (W)   // the weight from global memory (L2)
                                wa[j] = ld_readonly16(static_cast<const char *>(p.w) + (int64_t)((k * PC + j) * GT + t) * 16);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < PC; ++j) {
                    const int u = (k * PC + j) * GT + t;
                    const int so = (j * GT + t) * 16;
                    if constexpr (OUT == kOutT) {
                        if (u < nch) {
                            float a[V];
                            unpack(xa[j], a, T{});
                            float wv[V];
                            if constexpr (W) {
                                unpack(wa[j], wv, T{});
                            } else {
#pragma unroll
                                for (int e = 0; e < V; ++e) wv[e] = 1.f;
                            }
                            scale_out_pairs<WM>(a, r, wv, p.w_bias);
                            st16(static_cast<char *>(p.y) + roff + (int64_t)u * 16, pack(a, T{}));
                        }
                    } else {
                        // every lane joins its block's shuffles; `valid` is
                        // uniform over a block (rows are whole blocks)
                        const bool valid = u < nch;
                        float a[V], wv[V];
#pragma unroll
                        for (int e = 0; e < V; ++e) a[e] = 0.f, wv[e] = 1.f;
                        if (valid) {
                            unpack(lds16(xp + so), a, T{});
                            if constexpr (WR)
                                unpack(lds16(wp + so), wv, T{});
                            else if constexpr (W)
                                unpack(ld_readonly16(static_cast<const char *>(p.w) + (int64_t)u * 16), wv, T{});
                        }
                        scale_out_pairs<WM>(a, r, wv, p.w_bias);
                        store_quantised<V, OUT>(a, valid, p, row, u, t);
                    }
                }
                // the slot's next copy comes through the async proxy: order
                // this thread's shared-memory writes before it
                if constexpr (RES) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0 && ok) {
                    if (!(p.withhold && blockIdx.x == 0 && warp == 0 && qx + (unsigned)k == 0u))
                        mbar_arrive(&X.empty[xs]);
                    if (WR && !w_resident) mbar_arrive(&Wr.empty[ws]);
                }
                if (WR && !w_resident) ++qw;
            }
            qx += (unsigned)pieces;
        }
        if (!ok) s_failed = 1;
    }

    __syncthreads();
    if (s_failed && tid == 0) {
        atomicAdd(&g_tma_timeouts, 1u);
        // no copy may land after the block has left
        drain_ring(X, s_issued[0], p.wait_ns);
        if (RES) drain_ring(Rr, s_issued[1], p.wait_ns);
        if (WR) drain_ring(Wr, s_issued[2], p.wait_ns);
    }
}

}  // namespace rrn
