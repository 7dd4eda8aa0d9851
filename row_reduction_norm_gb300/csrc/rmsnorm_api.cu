// rmsnorm_api.cu -- the C ABI declared in include/rmsnorm.h: argument checks,
// host-side planning (which kernel, how many threads per row, grid size) and
// the launch.  No allocation, no synchronisation, the caller's stream.
//
// Planning follows the host-side decisions of "CuTeDSL at Perplexity":
// sections on the large configuration space (compile-time specialisation on
// dtype, weight / no weight and hidden size -- a branch that does not exist
// beats one that is always or never taken), on prefill vs decode (threads per
// block chosen from the token count, hidden size and SM count) and "Blackwell
// support" (the SM count is read from the device, not hard-coded).  The
// per-row schedule depends on hidden, dtype and alignment only; the row count
// only sizes the grid, so a row's result is the same in every batch.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kernel_table.h"
#include "layernorm_kernels.cuh"
#include "rmsnorm.h"
#include "rmsnorm_kernels.cuh"

static_assert(sizeof(rmsnorm_plan_t) == 48, "rmsnorm_plan_t layout is part of the ABI");

namespace {

constexpr int64_t kMaxHidden = 65536;
constexpr int64_t kRegTargetCH = 4;
// Row-group blocks beyond this many waves of resident blocks switch the grid
// to the persistent form (blocks stride over row groups).  Measured on GB300,
// one block per row group beats a grid capped at one wave for every workload
// up to 65536 x 8192, so the cap only engages for very large row counts.
constexpr int64_t kPersistentWaves = 4096;
constexpr int kMaxDevices = 64;
// Largest per-thread chain of squares the two-pass kernel may form (keeps the
// fp32 error bound of the sum the same as the register kernel's).
constexpr int64_t kLoopMaxTermsPerThread = 64;
// Dynamic shared memory of a register-kernel block with a weight: the weight
// row, at most kRegMaxGT * kRegMaxCH chunks of 16 bytes.
constexpr int kRegMaxWeightSmem = rrn::kRegMaxGT * rrn::kRegMaxCH * 16;
// Dynamic shared memory the bulk-copy kernel's ring may take: the 227 KB a
// block may opt in to on sm_103a, less 1 KB for the kernel's static arrays.
constexpr int kTmaSmemBudget = 227 * 1024 - 1024;
// Chunks per consumer thread per ring piece chosen by planning: 16 KB pieces
// (block-scaled outputs, fp32 rows up to 80 KB), and 32 KB pieces for bf16
// rows and rows past 80 KB (rows without a residual).
constexpr int kTmaPlanPC = 2;
constexpr int kTmaLongPC = 4;
// 16-byte units of a row past which contiguous RMSNorm rows leave the
// register kernel for the cluster kernel (with a residual) or the bulk-copy
// kernel (without one): 2048 units, 32 KB.
constexpr int64_t kRegWideUnits = 256 * rrn::kRegMaxCH;
// Limit of every wait inside the bulk-copy kernel (ns).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

int elem_size(int dtype) { return dtype == RMSNORM_BF16 ? 2 : 4; }
int vec_elems_of(int dtype) { return 16 / elem_size(dtype); }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t next_pow2(int64_t v) {
    int64_t p = 1;
    while (p < v) p <<= 1;
    return p;
}

bool aligned_to(const void *p, int a) {
    return p == nullptr || (reinterpret_cast<uintptr_t>(p) % (uintptr_t)a) == 0;
}

// Slots of the bulk-copy kernel's three rings (x, residual, weight).
struct TmaRings {
    int sx = 0, sr = 0, sw = 0;
};

// Ring sizes for rows of row_bytes with pieces of pc chunks a thread: the
// slots that fit the shared-memory budget are shared out as a streamed ring
// of avail / 7 slots (at least 1) for the residual; a weight ring holding the
// whole weight (one slot a piece) when the x ring still keeps a row and two
// spare slots beside it, else no weight ring (the kernel reads the weight
// from global memory: measured on GB300, bf16 2048 x 65536 without a residual
// 0.92 -> 0.96 of peak against a weight streamed through a ring, 2730 x 49152
// 0.93 -> 0.97 against a resident weight that left x one spare slot); the
// rest for x.  False when the x ring cannot hold a whole row.
bool tma_rings(int64_t row_bytes, int pc, bool res, bool w, TmaRings *out) {
    const int piece = rrn::tma_piece_bytes(pc);
    int avail = (kTmaSmemBudget - rrn::kTmaBarBytes) / piece;
    if (avail > rrn::kTmaMaxSlots) avail = rrn::kTmaMaxSlots;
    const int64_t pieces = ceil_div(row_bytes, piece);
    const int streamed = avail / 7 > 0 ? avail / 7 : 1;
    TmaRings R;
    R.sr = res ? streamed : 0;
    R.sw = (w && avail - R.sr - pieces >= pieces + 2) ? (int)pieces : 0;
    R.sx = avail - R.sr - R.sw;
    if (R.sx < pieces) return false;
    if (out) *out = R;
    return true;
}

// Everything one launch needs, for contiguous rows and for head rows.
struct Op {
    const void *x = nullptr, *res = nullptr, *w = nullptr, *w2 = nullptr;
    void *y = nullptr, *res_out = nullptr;
    int64_t rows = 0;          // launch rows: rows, or tokens * heads
    int64_t row_elems = 0;     // hidden or head_dim
    int64_t x_stride = 0;      // elements between rows (tokens for head rows)
    int64_t y_stride = 0;
    int32_t heads = 1, q_heads = 1;
    bool head_rows = false;
    bool ln = false;           // LayerNorm instead of RMSNorm
    const void *b = nullptr;   // LayerNorm bias
    bool mx = false;           // MXFP8 output: y holds E4M3 codes, scales the E8M0 scales
    bool nv = false;           // NVFP4 output: y holds packed E2M1 codes, scales the E4M3 scales
    void *scales = nullptr;
    float q_scale = 1.f;       // NVFP4 per-tensor scale
    float eps = 0.f, w_bias = 0.f;
    int wm = 0;                // rrn::WeightMode (RMSNorm) or rrn::AffineMode (LayerNorm)
    int dtype = RMSNORM_BF16;
    uint64_t wait_ns = kWaitLimitNs;   // bulk-copy kernel: limit of each wait
    int withhold = 0;                  // bulk-copy kernel: test of its bounded waits
};

// Threads per block of a register-kernel plan for this op.
int reg_block_of(const Op &o, int gt) { return o.ln ? rrn::ln_block_threads(gt) : rrn::reg_block_threads(gt); }

int max_threads_per_row(const Op &o) {
    return o.ln ? rrn::kLnMaxGT : (o.head_rows ? rrn::kRegMaxGTHeads : rrn::kRegMaxGT);
}

bool elem_aligned(const Op &o) {
    const int a = elem_size(o.dtype);
    return aligned_to(o.x, a) && aligned_to(o.res, a) && aligned_to(o.w, a) && aligned_to(o.w2, a) &&
           aligned_to(o.b, a) && aligned_to(o.y, a) && aligned_to(o.res_out, a);
}

// 16-byte units are possible when every pointer, the row size and the row
// strides are multiples of 16 bytes.
int vec_ok_of(const Op &o) {
    const int s = elem_size(o.dtype);
    return aligned_to(o.x, 16) && aligned_to(o.res, 16) && aligned_to(o.w, 16) && aligned_to(o.w2, 16) &&
           aligned_to(o.b, 16) && aligned_to(o.y, 16) && aligned_to(o.res_out, 16) && (o.row_elems * s) % 16 == 0 &&
           (o.x_stride * s) % 16 == 0 && (o.y_stride * s) % 16 == 0;
}

// The per-row schedule: everything but the grid (and, for contiguous
// RMSNorm rows, the exact-fit chunk count that fit_chunks picks from the row
// count).
// odd_ch: chunk counts 3 and 6 are chosen where they fit the row exactly
// (LayerNorm rows).
// tma_ok: the op has bulk-copy and cluster kernels (contiguous RMSNorm rows
// in the I/O type).  For these ops, measured on GB300: rows of 16 to 32 KB
// run best as 256 threads x 8 chunks (not 512 x 4), and longer rows on the
// cluster kernel with a residual and on the bulk-copy kernel without one
// (not 512 x 8 in registers); has_res matters only for rows past 32 KB.
void schedule(int64_t hidden, int dtype, int vec_ok, int max_gt, rmsnorm_plan_t *p, bool odd_ch = false,
              bool tma_ok = false, bool has_res = false) {
    std::memset(p, 0, sizeof(*p));
    const int V = vec_elems_of(dtype);
    if (vec_ok) {
        const int64_t nch = hidden / V;
        const int64_t row_bytes = hidden * elem_size(dtype);
        // Rows past 32 KB with a residual: the cluster kernel, a row over the
        // fewest blocks of 16 KB slices (32 KB slices for fp32 rows past 128
        // KB) -- measured on GB300 faster than the bulk-copy kernel (rows up
        // to 80 KB) and the two-pass kernel (longer rows) for every such row;
        // without a residual the bulk-copy kernel stays (below).  Rows that
        // five 16 KB slices would take (64 to 80 KB) take four of 20 KB:
        // bf16 4096 x 40960 0.976 of peak against 0.961.
        if (tma_ok && has_res && nch > kRegWideUnits) {
            int ch = 4;
            int64_t ctas = ceil_div(nch, (int64_t)rrn::kClusterGT * ch);
            if (ctas == 5) {
                ch = 5;
                ctas = ceil_div(nch, (int64_t)rrn::kClusterGT * ch);
            }
            if (ctas > rrn::kClusterMaxCtas && dtype == RMSNORM_F32) {
                ch = 8;
                ctas = ceil_div(nch, (int64_t)rrn::kClusterGT * ch);
            }
            if (ctas <= rrn::kClusterMaxCtas) {
                p->kernel = RMSNORM_KERNEL_CLUSTER;
                p->regime = RMSNORM_REGIME_CLUSTER;
                p->threads_per_row = rrn::kClusterGT * (int32_t)ctas;
                p->chunks_per_thread = ch;
                p->vec_elems = V;
                p->block_threads = rrn::kClusterGT;
                p->rows_per_block = 1;
                p->cluster_ctas = (int32_t)ctas;
                return;
            }
        }
        // Rows past 32 KB without a residual: the bulk-copy kernel, the
        // weight resident beside the row where that leaves x two spare slots
        // (rows up to 80 KB), else read from global memory while x keeps one
        // spare slot (rows up to 192 KB).  Pieces of 32 KB for bf16 rows and
        // rows past 80 KB, else 16 KB -- each the faster choice measured on
        // GB300.  The piece size changes no result; the kernel does.
        TmaRings tr;
        int tma_pc = 0;
        if (tma_ok && !has_res && nch > kRegWideUnits) {
            if (tma_rings(row_bytes, kTmaPlanPC, true, true, &tr) && tr.sw > 0)
                tma_pc = dtype == RMSNORM_BF16 ? kTmaLongPC : kTmaPlanPC;
            else if (tma_rings(row_bytes, kTmaLongPC, false, true, &tr) &&
                     tr.sx > ceil_div(row_bytes, rrn::tma_piece_bytes(kTmaLongPC)))
                tma_pc = kTmaLongPC;   // planned while x keeps a spare slot (rows up to 192 KB)
        }
        if (tma_pc > 0) {
            p->kernel = RMSNORM_KERNEL_TMA;
            p->regime = RMSNORM_REGIME_SMEM;
            p->threads_per_row = rrn::kTmaGT;
            p->chunks_per_thread = tma_pc;
            p->vec_elems = V;
            p->block_threads = rrn::kTmaBlock;
            p->rows_per_block = 1;
            return;
        }
        // Aim at 4 chunks (64 bytes of each input) per thread with at least 4
        // lanes per row: measured on GB300, this keeps every row-group block
        // resident in one wave at the occupancy the registers allow and beats
        // 8 chunks per thread.  Rows longer than max_gt threads x 4 chunks
        // take up to 8 chunks per thread.
        int64_t gt = next_pow2(ceil_div(nch, kRegTargetCH));
        if (gt < 4) gt = 4;
        if (gt > max_gt && ceil_div(nch, max_gt) <= rrn::kRegMaxCH) gt = max_gt;
        if (tma_ok && gt > 256 && ceil_div(nch, 256) <= rrn::kRegMaxCH) gt = 256;
        if (gt <= max_gt) {
            int64_t need = ceil_div(nch, gt);
            int ch = 1;
            while (ch < need) ch <<= 1;
            if (odd_ch && (need == 3 || need == 5 || need == 6)) ch = need == 3 ? 3 : 6;
            p->kernel = RMSNORM_KERNEL_REG;
            p->threads_per_row = (int32_t)gt;
            p->chunks_per_thread = ch;
            p->vec_elems = V;
            p->block_threads = rrn::reg_block_threads((int)gt);
            p->rows_per_block = p->block_threads / (int32_t)gt;
            p->regime = gt <= 32 ? RMSNORM_REGIME_WARP : RMSNORM_REGIME_CTA;
            return;
        }
    }
    p->kernel = RMSNORM_KERNEL_LOOP;
    p->vec_elems = vec_ok ? V : 1;
    const int64_t units = hidden / p->vec_elems;
    int block = rrn::kLoopBlocks[2];
    for (int b : rrn::kLoopBlocks) {
        if (ceil_div(units, b) * p->vec_elems <= kLoopMaxTermsPerThread) {
            block = b;
            break;
        }
    }
    p->block_threads = block;
    p->threads_per_row = block;
    p->chunks_per_thread = 0;
    p->rows_per_block = 1;
    p->regime = RMSNORM_REGIME_LOOPED;
}

void size_grid(int64_t rows, int sm_count, int blocks_per_sm, rmsnorm_plan_t *p) {
    const int64_t row_blocks = ceil_div(rows, p->rows_per_block);
    const int64_t resident = (int64_t)(sm_count > 0 ? sm_count : 1) * (blocks_per_sm > 0 ? blocks_per_sm : 1);
    p->pdl = 1;
    if (p->kernel == RMSNORM_KERNEL_CLUSTER) {   // one cluster a row
        const int64_t cap = INT_MAX / (p->cluster_ctas > 0 ? p->cluster_ctas : 1);
        const int64_t clusters = rows < cap ? rows : cap;
        p->grid = clusters * p->cluster_ctas;
        p->persistent = rows > clusters;
        return;
    }
    if (p->kernel == RMSNORM_KERNEL_TMA) {   // one wave; blocks stride over the rows
        p->grid = row_blocks < resident ? row_blocks : resident;
        p->persistent = row_blocks > p->grid;
        return;
    }
    int64_t cap = resident * kPersistentWaves;
    if (cap > INT_MAX) cap = INT_MAX;
    p->persistent = row_blocks > cap;
    p->grid = row_blocks > cap ? cap : row_blocks;
    p->pdl = 1;
    if (p->persistent && p->kernel == RMSNORM_KERNEL_REG) p->regime = RMSNORM_REGIME_PERSISTENT;
}

// Chunk count that fits a register-kernel row exactly (3 or 6 chunks where
// the power of two would leave slots idle).  Chunks past the row end add exact
// zeros to the sum, so any count that covers the row gives the same result.
int exact_ch(int64_t units, int gt, int ch) {
    const int64_t need = ceil_div(units, gt);
    if (need == 3) return 3;
    if (need == 5 || need == 6) return 6;
    return ch;
}

// Contiguous RMSNorm rows take the exact-fit chunk count when the launch has
// more than one wave of blocks, and always for rows of a warp or less:
// measured on GB300 it is faster there (fewer registers, more blocks
// resident: bf16 233016 x 576 without residual 0.874 -> 0.985 of peak,
// 26214 x 5120 0.855 -> 0.983; with the first rows prefetched before the
// dependency wait, a single wave of bf16 rows of 576 too: 4096 rows 2.31 ->
// 2.18 us, 1024 rows 1.77 -> 1.70 us), but not for a single wave of wider
// rows (bf16 600 x 5120: 2.85 us with 4 chunks against 3.01 with 3).
void fit_chunks(int64_t rows, int64_t resident_blocks, bool contiguous_rms, int64_t units, rmsnorm_plan_t *p) {
    if (!contiguous_rms || p->kernel != RMSNORM_KERNEL_REG) return;
    if (p->threads_per_row > 32 && ceil_div(rows, p->rows_per_block) <= resident_blocks) return;
    p->chunks_per_thread = exact_ch(units, p->threads_per_row, p->chunks_per_thread);
}

// Decode batches -- launches whose rows fit in one warp of row slots a block
// without needing more blocks than the device has SMs -- hold one warp of
// rows a block (one row for rows of a warp or more, 32 / threads_per_row
// rows below), so the rows spread over as many SMs as they can (the register
// kernel takes a run-time count of rows a block; the idle row slots load and
// store nothing).  The page's decode variant is one warp a block while fewer
// warps than SMs are needed; measured on GB300: bf16 rows of 4096, 8 rows
// 1.66 -> 1.62 us, 64 rows 1.82 -> 1.71 us; rows of 576, 8 rows 1.45 -> 1.34
// us, 64 rows 1.53 -> 1.38 us; fp32 64 x 256 (16 threads a row) 1.40 -> 1.26
// us; bf16 64 x 128 (4 threads a row) 1.48 -> 1.27 us; a single row the same.
// The per-row schedule is unchanged, so no result changes.  Planned for
// contiguous RMSNorm rows (what was measured); forced plans may hold fewer
// rows a block on every RMSNorm register kernel.
void spread_rows(int64_t rows, int sm_count, bool contiguous_rms, rmsnorm_plan_t *p) {
    if (!contiguous_rms || p->kernel != RMSNORM_KERNEL_REG) return;
    const int gt = p->threads_per_row;
    const int want = gt >= 32 ? 1 : 32 / gt;   // one warp of rows a block
    if (want >= p->rows_per_block || rows < 1) return;
    const int64_t blocks = ceil_div(rows, want);
    if (blocks > (int64_t)(sm_count > 0 ? sm_count : 1)) return;
    p->rows_per_block = want;
    p->grid = blocks;
    p->persistent = 0;
    if (p->regime == RMSNORM_REGIME_PERSISTENT) p->regime = gt <= 32 ? RMSNORM_REGIME_WARP : RMSNORM_REGIME_CTA;
}

size_t dyn_smem_of(const rmsnorm_plan_t *p, const Op &o) {
    if (p->kernel == RMSNORM_KERNEL_TMA) {
        TmaRings R;
        if (!tma_rings(o.row_elems * elem_size(o.dtype), p->chunks_per_thread, o.res != nullptr, o.w != nullptr, &R))
            return 0;
        return (size_t)rrn::tma_smem_bytes(p->chunks_per_thread, R.sx + R.sr + R.sw);
    }
    if (p->kernel != RMSNORM_KERNEL_REG || o.wm == 0) return 0;
    const int copies = o.ln ? (o.wm == rrn::kAffWB ? 2 : 1) : (o.head_rows ? 2 : 1);
    return (size_t)(o.row_elems / vec_elems_of(o.dtype)) * 16 * copies;
}

// Smallest row group of the MXFP8 form: the lanes of one 32-element block.
int mx_min_gt(int dtype) { return 32 / vec_elems_of(dtype); }

const void *kernel_of(const rmsnorm_plan_t *p, const Op &o) {
    const bool res = o.res != nullptr;
    if (p->kernel == RMSNORM_KERNEL_CLUSTER) {
        if (o.ln || o.head_rows || o.mx || o.nv) return nullptr;
        return rrn::cluster_kernel(o.dtype, p->chunks_per_thread, res, o.wm);
    }
    if (p->kernel == RMSNORM_KERNEL_TMA) {
        if (o.ln || o.head_rows) return nullptr;
        // the weight from global memory when the rings give it no slots
        TmaRings R;
        if (!tma_rings(o.row_elems * elem_size(o.dtype), p->chunks_per_thread, res, o.w != nullptr, &R))
            return nullptr;
        const bool wg = o.w != nullptr && R.sw == 0;
        if (o.mx || o.nv)
            return p->chunks_per_thread == 2 ? rrn::tma_quant_kernel(o.dtype, res, o.wm, o.mx ? rrn::kOutMxfp8
                                                                                              : rrn::kOutNvfp4, wg)
                                             : nullptr;
        return rrn::tma_kernel(o.dtype, p->chunks_per_thread, res, o.wm, wg);
    }
    if (o.mx || o.nv) {
        if (p->kernel != RMSNORM_KERNEL_REG) return nullptr;
        return o.mx ? rrn::mx_kernel(o.dtype, p->threads_per_row, p->chunks_per_thread, res, o.wm)
                    : rrn::nv_kernel(o.dtype, p->threads_per_row, p->chunks_per_thread, res, o.wm);
    }
    if (o.ln) {
        if (p->kernel == RMSNORM_KERNEL_REG)
            return o.dtype == RMSNORM_BF16 ? rrn::ln_reg_bf16(p->threads_per_row, p->chunks_per_thread, res, o.wm)
                                           : rrn::ln_reg_f32(p->threads_per_row, p->chunks_per_thread, res, o.wm);
        return rrn::ln_loop(o.dtype, p->block_threads, p->vec_elems != 1, res, o.wm);
    }
    if (o.wm == rrn::kWeightCast) {
        if (o.dtype != RMSNORM_BF16 || o.head_rows) return nullptr;
        if (p->kernel == RMSNORM_KERNEL_REG)
            return rrn::reg_contig_bf16_cast(p->threads_per_row, p->chunks_per_thread, res);
        return rrn::loop_contig_bf16_cast(p->block_threads, p->vec_elems != 1, res);
    }
    if (p->kernel == RMSNORM_KERNEL_REG)
        return rrn::reg_kernel(o.dtype, p->threads_per_row, p->chunks_per_thread, res, o.wm, o.head_rows);
    return rrn::loop_kernel(o.dtype, p->block_threads, p->vec_elems != 1, res, o.wm, o.head_rows);
}

// Checks a plan against the shape and pointers (caller-made plans included).
int validate_plan(const rmsnorm_plan_t *p, const Op &o, int vec_ok) {
    if (p == nullptr) return RMSNORM_EINVAL;
    const int V = vec_elems_of(o.dtype);
    if (o.rows > 0 && (p->grid < 1 || p->grid > INT_MAX)) return RMSNORM_EINVAL;
    if (p->pdl != 0 && p->pdl != 1) return RMSNORM_EINVAL;
    if (p->kernel != RMSNORM_KERNEL_CLUSTER && p->cluster_ctas != 0) return RMSNORM_EINVAL;
    if (p->kernel == RMSNORM_KERNEL_REG) {
        const int gt = p->threads_per_row, ch = p->chunks_per_thread;
        const int max_gt = max_threads_per_row(o);
        if (!vec_ok || p->vec_elems != V) return RMSNORM_EINVAL;
        if (gt < 4 || gt > max_gt || (gt & (gt - 1)) != 0) return RMSNORM_EINVAL;
        if (o.mx && gt < mx_min_gt(o.dtype)) return RMSNORM_EINVAL;
        const bool odd_ch = ch == 3 || ch == 6;   // compiled for contiguous RMSNorm / LayerNorm rows
        if (ch < 1 || ch > rrn::kRegMaxCH || ((ch & (ch - 1)) != 0 && !odd_ch)) return RMSNORM_EINVAL;
        if (odd_ch && (o.head_rows || o.mx || o.nv)) return RMSNORM_EINVAL;
        if ((int64_t)gt * ch * V < o.row_elems) return RMSNORM_EINVAL;
        if (p->block_threads != reg_block_of(o, gt)) return RMSNORM_EINVAL;
        // LayerNorm blocks hold every row slot; the RMSNorm kernel may hold fewer
        if (o.ln ? p->rows_per_block != p->block_threads / gt
                 : (p->rows_per_block < 1 || p->rows_per_block > p->block_threads / gt))
            return RMSNORM_EINVAL;
        return RMSNORM_OK;
    }
    if (p->kernel == RMSNORM_KERNEL_CLUSTER) {
        // contiguous RMSNorm rows with a residual, in the I/O type
        if (o.ln || o.head_rows || o.mx || o.nv || o.res == nullptr) return RMSNORM_EINVAL;
        if (!vec_ok || p->vec_elems != V) return RMSNORM_EINVAL;
        const int ch = p->chunks_per_thread, c = p->cluster_ctas;
        if (rrn::cluster_kernel(o.dtype, ch, true, o.wm) == nullptr) return RMSNORM_EINVAL;   // not compiled
        if (c < 2 || c > rrn::kClusterMaxCtas) return RMSNORM_EINVAL;
        if (p->block_threads != rrn::kClusterGT || p->threads_per_row != rrn::kClusterGT * c ||
            p->rows_per_block != 1)
            return RMSNORM_EINVAL;
        if ((int64_t)c * rrn::kClusterGT * ch * V < o.row_elems) return RMSNORM_EINVAL;
        if (o.rows > 0 && p->grid % c != 0) return RMSNORM_EINVAL;
        return RMSNORM_OK;
    }
    if (p->kernel == RMSNORM_KERNEL_TMA) {
        if (o.ln || o.head_rows) return RMSNORM_EINVAL;   // contiguous RMSNorm rows only
        if ((o.mx || o.nv) && p->chunks_per_thread != 2) return RMSNORM_EINVAL;   // compiled for 16 KB pieces
        if (!vec_ok || p->vec_elems != V) return RMSNORM_EINVAL;
        if (p->threads_per_row != rrn::kTmaGT || p->block_threads != rrn::kTmaBlock || p->rows_per_block != 1)
            return RMSNORM_EINVAL;
        const int pc = p->chunks_per_thread;
        if (pc != 1 && pc != 2 && pc != 4) return RMSNORM_EINVAL;
        if (!tma_rings(o.row_elems * elem_size(o.dtype), pc, o.res != nullptr, o.w != nullptr, nullptr))
            return RMSNORM_EINVAL;
        return RMSNORM_OK;
    }
    if (p->kernel == RMSNORM_KERNEL_LOOP) {
        if (o.mx || o.nv) return RMSNORM_EINVAL;   // block-scaled forms run on the register kernel only
        if (p->vec_elems != 1 && !(p->vec_elems == V && vec_ok)) return RMSNORM_EINVAL;
        bool known = false;
        for (int b : rrn::kLoopBlocks) known = known || (b == p->block_threads);
        if (!known) return RMSNORM_EINVAL;
        if (p->rows_per_block != 1) return RMSNORM_EINVAL;
        if (ceil_div(o.row_elems / p->vec_elems, p->block_threads) * p->vec_elems > kLoopMaxTermsPerThread)
            return RMSNORM_EINVAL;
        return RMSNORM_OK;
    }
    return RMSNORM_EINVAL;
}

// ------------------------------------------------------------ device caches

std::mutex g_mu;
int g_sm_count[kMaxDevices];

struct OccEntry {
    int dev;
    const void *fn;
    size_t smem;
    int blocks;
};
constexpr int kOccSlots = 1024;
OccEntry g_occ[kOccSlots];
int g_occ_used = 0;

struct AttrEntry {
    int dev;
    const void *fn;
};
AttrEntry g_attr[kOccSlots];
int g_attr_used = 0;

int sm_count_of(int dev, int *out) {
    if (dev < 0 || dev >= kMaxDevices) return RMSNORM_ECUDA;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_sm_count[dev] > 0) {
            *out = g_sm_count[dev];
            return RMSNORM_OK;
        }
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return RMSNORM_ECUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    g_sm_count[dev] = n;
    *out = n;
    return RMSNORM_OK;
}

// Opt a kernel in to the largest dynamic shared memory its family may be
// given (the weight row of the register kernel, the bulk-copy kernel's ring).
int ensure_smem_attr(int dev, const void *fn, const rmsnorm_plan_t *p) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_attr_used; ++i)
        if (g_attr[i].dev == dev && g_attr[i].fn == fn) return RMSNORM_OK;
    const int bytes = p->kernel == RMSNORM_KERNEL_TMA ? kTmaSmemBudget : kRegMaxWeightSmem;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return RMSNORM_ECUDA;
    if (g_attr_used < kOccSlots) g_attr[g_attr_used++] = AttrEntry{dev, fn};
    return RMSNORM_OK;
}

int blocks_per_sm_of(int dev, const void *fn, int block, size_t smem, int *out) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int i = 0; i < g_occ_used; ++i) {
            if (g_occ[i].dev == dev && g_occ[i].fn == fn && g_occ[i].smem == smem) {
                *out = g_occ[i].blocks;
                return RMSNORM_OK;
            }
        }
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, block, smem) != cudaSuccess || n <= 0)
        return RMSNORM_ECUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_occ_used < kOccSlots) g_occ[g_occ_used++] = OccEntry{dev, fn, smem, n};
    *out = n;
    return RMSNORM_OK;
}

// Full device-side planning for an op.
int plan_for_device(const Op &o, rmsnorm_plan_t *plan, int *dev_out) {
    schedule(o.row_elems, o.dtype, vec_ok_of(o), max_threads_per_row(o), plan, o.ln,
             !(o.ln || o.head_rows || o.mx || o.nv), o.res != nullptr);
    if ((o.mx || o.nv) && plan->kernel != RMSNORM_KERNEL_REG) {
        // rows too long for registers: the bulk-copy kernel with 16 KB pieces
        // when its rings hold the row, else unsupported
        if (!vec_ok_of(o) ||
            !tma_rings(o.row_elems * elem_size(o.dtype), kTmaPlanPC, o.res != nullptr, o.w != nullptr, nullptr))
            return RMSNORM_EUNSUPPORTED;
        std::memset(plan, 0, sizeof(*plan));
        plan->kernel = RMSNORM_KERNEL_TMA;
        plan->regime = RMSNORM_REGIME_SMEM;
        plan->threads_per_row = rrn::kTmaGT;
        plan->chunks_per_thread = kTmaPlanPC;
        plan->vec_elems = vec_elems_of(o.dtype);
        plan->block_threads = rrn::kTmaBlock;
        plan->rows_per_block = 1;
    }
    if (o.ln && plan->kernel == RMSNORM_KERNEL_REG) {
        plan->block_threads = reg_block_of(o, plan->threads_per_row);
        plan->rows_per_block = plan->block_threads / plan->threads_per_row;
    }
    if (o.mx && plan->kernel == RMSNORM_KERNEL_REG) {
        const int V = vec_elems_of(o.dtype);
        while (plan->threads_per_row < mx_min_gt(o.dtype)) plan->threads_per_row <<= 1;
        int64_t need = ceil_div(o.row_elems / V, plan->threads_per_row);
        int ch = 1;
        while (ch < need) ch <<= 1;
        plan->chunks_per_thread = ch;
        plan->block_threads = rrn::reg_block_threads(plan->threads_per_row);
        plan->rows_per_block = plan->block_threads / plan->threads_per_row;
        plan->regime = plan->threads_per_row <= 32 ? RMSNORM_REGIME_WARP : RMSNORM_REGIME_CTA;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RMSNORM_ECUDA;
    int sms = 0;
    int st = sm_count_of(dev, &sms);
    if (st != RMSNORM_OK) return st;
    const void *fn = kernel_of(plan, o);
    if (fn == nullptr) return RMSNORM_EINVAL;
    const size_t smem = dyn_smem_of(plan, o);
    if (smem > 0 && (st = ensure_smem_attr(dev, fn, plan)) != RMSNORM_OK) return st;
    int bps = 0;
    if ((st = blocks_per_sm_of(dev, fn, plan->block_threads, smem, &bps)) != RMSNORM_OK) return st;
    size_grid(o.rows, sms, bps, plan);
    fit_chunks(o.rows, (int64_t)sms * bps, !(o.ln || o.head_rows || o.mx || o.nv), o.row_elems / vec_elems_of(o.dtype),
               plan);
    spread_rows(o.rows, sms, !(o.ln || o.head_rows || o.mx || o.nv), plan);
    if (dev_out) *dev_out = dev;
    return RMSNORM_OK;
}

int launch(const Op &o, const rmsnorm_plan_t *plan, int dev, rmsnorm_stream_t stream) {
    const void *fn = kernel_of(plan, o);
    if (fn == nullptr) return RMSNORM_EINVAL;
    const size_t smem = dyn_smem_of(plan, o);
    if (smem > 0) {
        int st = ensure_smem_attr(dev, fn, plan);
        if (st != RMSNORM_OK) return st;
    }
    const int64_t s = elem_size(o.dtype);
    rrn::Params args;
    rrn::LnParams largs;
    TmaRings rings;
    void *argv[4];
    if (o.ln) {
        largs.x = o.x;
        largs.res = o.res;
        largs.w = o.w;
        largs.b = o.b;
        largs.y = o.y;
        largs.res_out = o.res_out;
        largs.rows = o.rows;
        largs.row_elems = o.row_elems;
        largs.row_bytes = o.row_elems * s;
        largs.units = (int32_t)(o.row_elems / plan->vec_elems);
        largs.hidden_f = (float)o.row_elems;
        largs.eps = o.eps;
        argv[0] = &largs;
    } else {
        argv[0] = &args;
    }
    args.x = o.x;
    args.res = o.res;
    args.w = o.w;
    args.w2 = o.w2;
    args.y = o.y;
    args.res_out = o.res_out;
    args.rows = o.rows;
    args.row_elems = o.row_elems;
    args.row_bytes = o.row_elems * s;
    args.x_stride = o.x_stride * s;
    args.y_stride = o.y_stride * s;
    args.units = (int32_t)(o.row_elems / plan->vec_elems);
    args.heads = o.heads;
    args.q_heads = o.q_heads;
    args.hidden_f = (float)o.row_elems;
    args.eps = o.eps;
    args.w_bias = o.w_bias;
    args.scales = o.scales;
    args.q_scale = o.q_scale;
    args.q_inv6s = (float)(1.0 / (6.0 * (double)o.q_scale));
    args.rpb = plan->rows_per_block;
    args.wait_ns = o.wait_ns;
    args.withhold = o.withhold;
    if (plan->kernel == RMSNORM_KERNEL_TMA) {
        if (!tma_rings(o.row_elems * s, plan->chunks_per_thread, o.res != nullptr, o.w != nullptr, &rings))
            return RMSNORM_EINVAL;
        argv[1] = &rings.sx;
        argv[2] = &rings.sr;
        argv[3] = &rings.sw;
    }
    cudaLaunchAttribute attr[2];
    unsigned nattr = 0;
    if (plan->pdl) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    if (plan->kernel == RMSNORM_KERNEL_CLUSTER) {   // blocks q*C .. q*C + C - 1 form cluster q
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = (unsigned)plan->cluster_ctas;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan->grid);
    cfg.blockDim = dim3((unsigned)plan->block_threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, argv);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();   // clear the non-sticky launch error
        return RMSNORM_ECUDA;
    }
    return RMSNORM_OK;
}

// Plan (if none is given), validate and launch.
int run(const Op &o, const rmsnorm_plan_t *user_plan, rmsnorm_stream_t stream) {
    if (!elem_aligned(o)) return RMSNORM_EINVAL;
    const int vec_ok = vec_ok_of(o);
    if (user_plan != nullptr) {
        int st = validate_plan(user_plan, o, vec_ok);
        if (st != RMSNORM_OK) return st;
    }
    if (o.rows == 0) return RMSNORM_OK;
    rmsnorm_plan_t plan;
    int dev = 0;
    if (user_plan == nullptr) {
        int st = plan_for_device(o, &plan, &dev);
        if (st != RMSNORM_OK) return st;
    } else {
        plan = *user_plan;
        if (cudaGetDevice(&dev) != cudaSuccess) return RMSNORM_ECUDA;
    }
    return launch(o, &plan, dev, stream);
}

int check_common(int64_t rows, int64_t row_elems, float eps, float w_bias, int dtype) {
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16) return RMSNORM_EINVAL;
    if (rows < 0 || row_elems <= 0) return RMSNORM_EINVAL;
    if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(w_bias)) return RMSNORM_EINVAL;
    if (row_elems > kMaxHidden) return RMSNORM_EUNSUPPORTED;
    return RMSNORM_OK;
}

int make_contig(const void *x, const void *residual, const void *w, void *y, void *residual_out, int64_t rows,
                int64_t hidden, float eps, float w_bias, int dtype, Op *o) {
    int st = check_common(rows, hidden, eps, w_bias, dtype);
    if (st != RMSNORM_OK) return st;
    if (rows > INT64_MAX / (hidden * elem_size(dtype))) return RMSNORM_EINVAL;
    if (rows > 0) {
        if (x == nullptr || y == nullptr) return RMSNORM_EINVAL;
        if ((residual == nullptr) != (residual_out == nullptr)) return RMSNORM_EINVAL;
    }
    if (w_bias != 0.f && w == nullptr) return RMSNORM_EINVAL;
    o->x = x;
    o->res = residual;
    o->w = w;
    o->y = y;
    o->res_out = residual_out;
    o->rows = rows;
    o->row_elems = hidden;
    o->x_stride = hidden;
    o->y_stride = hidden;
    o->eps = eps;
    o->w_bias = w_bias;
    o->wm = w == nullptr ? rrn::kNoWeight : (w_bias != 0.f ? rrn::kWeightBias : rrn::kWeight);
    o->dtype = dtype;
    return RMSNORM_OK;
}

int make_heads(const void *x, void *y, int64_t tokens, int64_t x_token_stride, int64_t y_token_stride,
               int32_t q_heads, int32_t k_heads, int64_t head_dim, const void *q_w, const void *k_w, float w_bias,
               float eps, int dtype, Op *o) {
    int st = check_common(tokens, head_dim, eps, w_bias, dtype);
    if (st != RMSNORM_OK) return st;
    if (q_heads < 0 || k_heads < 0 || (int64_t)q_heads + k_heads < 1 || (int64_t)q_heads + k_heads > INT_MAX)
        return RMSNORM_EINVAL;
    const int64_t heads = (int64_t)q_heads + k_heads;
    const int64_t span = heads * head_dim;
    if (x_token_stride < span || y_token_stride < span) return RMSNORM_EINVAL;
    const int64_t s = elem_size(dtype);
    const int64_t big = x_token_stride > y_token_stride ? x_token_stride : y_token_stride;
    if (tokens > INT64_MAX / (big * s) || tokens > INT64_MAX / heads) return RMSNORM_EINVAL;
    if ((q_w == nullptr) != (k_w == nullptr)) return RMSNORM_EINVAL;
    if (w_bias != 0.f && q_w == nullptr) return RMSNORM_EINVAL;
    if (tokens > 0 && (x == nullptr || y == nullptr)) return RMSNORM_EINVAL;
    if (x == y && x_token_stride != y_token_stride) return RMSNORM_EINVAL;
    o->x = x;
    o->y = y;
    o->w = q_w;
    o->w2 = k_w;
    o->rows = tokens * heads;
    o->row_elems = head_dim;
    o->x_stride = x_token_stride;
    o->y_stride = y_token_stride;
    o->heads = (int32_t)heads;
    o->q_heads = q_heads;
    o->head_rows = true;
    o->eps = eps;
    o->w_bias = w_bias;
    o->wm = q_w == nullptr ? rrn::kNoWeight : (w_bias != 0.f ? rrn::kWeightBias : rrn::kWeight);
    o->dtype = dtype;
    return RMSNORM_OK;
}

int make_mx(const void *x, const void *residual, const void *w, void *codes, void *scales, void *residual_out,
            int64_t rows, int64_t hidden, float eps, float w_bias, int dtype, Op *o) {
    int st = make_contig(x, residual, w, codes, residual_out, rows, hidden, eps, w_bias, dtype, o);
    if (st != RMSNORM_OK) return st;
    if (hidden % 32 != 0) return RMSNORM_EINVAL;
    if (rows > 0 && scales == nullptr) return RMSNORM_EINVAL;
    o->mx = true;
    o->scales = scales;
    // the codes are bytes: their row stride is hidden bytes, which the register
    // kernel derives from row_elems; y_stride (in elements of T) is unused
    return RMSNORM_OK;
}

int make_nv(const void *x, const void *residual, const void *w, void *codes, void *scales, void *residual_out,
            int64_t rows, int64_t hidden, float eps, float w_bias, float tensor_scale, int dtype, Op *o) {
    int st = make_contig(x, residual, w, codes, residual_out, rows, hidden, eps, w_bias, dtype, o);
    if (st != RMSNORM_OK) return st;
    if (hidden % 16 != 0) return RMSNORM_EINVAL;
    if (!(tensor_scale > 0.f) || !std::isfinite(tensor_scale)) return RMSNORM_EINVAL;
    if (dtype != RMSNORM_BF16) return RMSNORM_EUNSUPPORTED;
    if (rows > 0 && scales == nullptr) return RMSNORM_EINVAL;
    o->nv = true;
    o->scales = scales;
    o->q_scale = tensor_scale;
    return RMSNORM_OK;
}

int make_ln(const void *x, const void *residual, const void *w, const void *b, void *y, void *residual_out,
            int64_t rows, int64_t hidden, float eps, int dtype, Op *o) {
    int st = make_contig(x, residual, w, y, residual_out, rows, hidden, eps, 0.f, dtype, o);
    if (st != RMSNORM_OK) return st;
    if (b != nullptr && w == nullptr) return RMSNORM_EINVAL;
    o->ln = true;
    o->b = b;
    o->wm = w == nullptr ? rrn::kAffNone : (b == nullptr ? rrn::kAffW : rrn::kAffWB);
    return RMSNORM_OK;
}

}  // namespace

extern "C" {

int rmsnorm_fwd_mxfp8(const void *x, const void *residual, const void *w, void *codes, void *scales,
                      void *residual_out, int64_t rows, int64_t hidden, float eps, float weight_bias, int dtype,
                      const rmsnorm_plan_t *plan, rmsnorm_stream_t stream) {
    Op o;
    int st = make_mx(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias, dtype, &o);
    if (st != RMSNORM_OK) return st;
    if (rows > 0 && !vec_ok_of(o)) return RMSNORM_EINVAL;   // 16-byte aligned rows required
    return run(o, plan, stream);
}

int rmsnorm_fwd_nvfp4(const void *x, const void *residual, const void *w, void *codes, void *scales,
                      void *residual_out, int64_t rows, int64_t hidden, float eps, float weight_bias,
                      float tensor_scale, int dtype, const rmsnorm_plan_t *plan, rmsnorm_stream_t stream) {
    Op o;
    int st = make_nv(x, residual, w, codes, scales, residual_out, rows, hidden, eps, weight_bias, tensor_scale,
                     dtype, &o);
    if (st != RMSNORM_OK) return st;
    if (rows > 0 && !vec_ok_of(o)) return RMSNORM_EINVAL;   // 16-byte aligned rows required
    return run(o, plan, stream);
}

int rmsnorm_nvfp4_plan_for(const void *x, const void *residual, const void *w, const void *codes,
                           const void *scales, const void *residual_out, int64_t rows, int64_t hidden, int dtype,
                           rmsnorm_plan_t *plan) {
    if (plan == nullptr) return RMSNORM_EINVAL;
    Op o;
    int st = make_nv(x, residual, w, const_cast<void *>(codes), const_cast<void *>(scales),
                     const_cast<void *>(residual_out), rows, hidden, 0.f, 0.f, 1.f, dtype, &o);
    if (st != RMSNORM_OK) return st;
    if (!elem_aligned(o) || !vec_ok_of(o)) return RMSNORM_EINVAL;
    return plan_for_device(o, plan, nullptr);
}

int rmsnorm_mxfp8_plan_for(const void *x, const void *residual, const void *w, const void *codes,
                           const void *scales, const void *residual_out, int64_t rows, int64_t hidden, int dtype,
                           rmsnorm_plan_t *plan) {
    if (plan == nullptr) return RMSNORM_EINVAL;
    Op o;
    int st = make_mx(x, residual, w, const_cast<void *>(codes), const_cast<void *>(scales),
                     const_cast<void *>(residual_out), rows, hidden, 0.f, 0.f, dtype, &o);
    if (st != RMSNORM_OK) return st;
    if (!elem_aligned(o) || !vec_ok_of(o)) return RMSNORM_EINVAL;
    return plan_for_device(o, plan, nullptr);
}

int layernorm_fwd(const void *x, const void *residual, const void *w, const void *b, void *y, void *residual_out,
                  int64_t rows, int64_t hidden, float eps, int dtype, const rmsnorm_plan_t *plan,
                  rmsnorm_stream_t stream) {
    Op o;
    int st = make_ln(x, residual, w, b, y, residual_out, rows, hidden, eps, dtype, &o);
    if (st != RMSNORM_OK) return st;
    return run(o, plan, stream);
}

int layernorm_plan_for(const void *x, const void *residual, const void *w, const void *b, const void *y,
                       const void *residual_out, int64_t rows, int64_t hidden, int dtype, rmsnorm_plan_t *plan) {
    if (plan == nullptr) return RMSNORM_EINVAL;
    Op o;
    int st = make_ln(x, residual, w, b, const_cast<void *>(y), const_cast<void *>(residual_out), rows, hidden, 0.f,
                     dtype, &o);
    if (st != RMSNORM_OK) return st;
    if (!elem_aligned(o)) return RMSNORM_EINVAL;
    return plan_for_device(o, plan, nullptr);
}

int rmsnorm_plan(int64_t rows, int64_t hidden, int dtype, int vec_ok, int sm_count, int blocks_per_sm,
                 rmsnorm_plan_t *plan) {
    return rmsnorm_plan_ex(rows, hidden, dtype, vec_ok, 0, sm_count, blocks_per_sm, plan);
}

int rmsnorm_plan_ex(int64_t rows, int64_t hidden, int dtype, int vec_ok, int has_residual, int sm_count,
                    int blocks_per_sm, rmsnorm_plan_t *plan) {
    if (plan == nullptr || dtype < RMSNORM_F32 || dtype > RMSNORM_BF16 || rows < 0 || hidden <= 0)
        return RMSNORM_EINVAL;
    if (has_residual != 0 && has_residual != 1) return RMSNORM_EINVAL;
    if (hidden > kMaxHidden) return RMSNORM_EUNSUPPORTED;
    if (vec_ok && (hidden * elem_size(dtype)) % 16 != 0) return RMSNORM_EINVAL;
    schedule(hidden, dtype, vec_ok ? 1 : 0, rrn::kRegMaxGT, plan, false, true, has_residual == 1);
    size_grid(rows, sm_count, blocks_per_sm, plan);
    fit_chunks(rows, (int64_t)(sm_count > 0 ? sm_count : 1) * (blocks_per_sm > 0 ? blocks_per_sm : 1), true,
               hidden / vec_elems_of(dtype), plan);
    spread_rows(rows, sm_count, true, plan);
    return RMSNORM_OK;
}

int rmsnorm_regime(int64_t rows, int64_t hidden, int dtype) {
    // A stand-in address for 16-byte aligned tensors: planning reads no
    // pointer, it only looks at the alignment of each one.
    alignas(16) static const unsigned char kAligned[16] = {0};
    Op o;
    int st = make_contig(kAligned, nullptr, kAligned, const_cast<unsigned char *>(kAligned), nullptr, rows, hidden,
                         0.f, 0.f, dtype, &o);
    if (st != RMSNORM_OK) return st;
    rmsnorm_plan_t plan;
    if ((st = plan_for_device(o, &plan, nullptr)) != RMSNORM_OK) return st;
    return plan.regime;
}

int rmsnorm_plan_for(const void *x, const void *residual, const void *w, const void *y,
                     const void *residual_out, int64_t rows, int64_t hidden, int dtype,
                     rmsnorm_plan_t *plan) {
    if (plan == nullptr) return RMSNORM_EINVAL;
    Op o;
    int st = make_contig(x, residual, w, const_cast<void *>(y), const_cast<void *>(residual_out), rows, hidden,
                         0.f, 0.f, dtype, &o);
    if (st != RMSNORM_OK) return st;
    if (!elem_aligned(o)) return RMSNORM_EINVAL;
    return plan_for_device(o, plan, nullptr);
}

int rmsnorm_fwd(const void *x, const void *residual, const void *w, void *y, void *residual_out,
                int64_t rows, int64_t hidden, float eps, int dtype, rmsnorm_stream_t stream) {
    Op o;
    int st = make_contig(x, residual, w, y, residual_out, rows, hidden, eps, 0.f, dtype, &o);
    if (st != RMSNORM_OK) return st;
    return run(o, nullptr, stream);
}

int rmsnorm_fwd_plan(const void *x, const void *residual, const void *w, void *y, void *residual_out,
                     int64_t rows, int64_t hidden, float eps, int dtype, const rmsnorm_plan_t *plan,
                     rmsnorm_stream_t stream) {
    if (plan == nullptr) return RMSNORM_EINVAL;
    Op o;
    int st = make_contig(x, residual, w, y, residual_out, rows, hidden, eps, 0.f, dtype, &o);
    if (st != RMSNORM_OK) return st;
    return run(o, plan, stream);
}

int rmsnorm_fwd_ex(const void *x, const void *residual, const void *w, void *y, void *residual_out,
                   int64_t rows, int64_t hidden, float eps, float weight_bias, int dtype,
                   const rmsnorm_plan_t *plan, rmsnorm_stream_t stream) {
    Op o;
    int st = make_contig(x, residual, w, y, residual_out, rows, hidden, eps, weight_bias, dtype, &o);
    if (st != RMSNORM_OK) return st;
    return run(o, plan, stream);
}

int rmsnorm_fwd_cast(const void *x, const void *residual, const void *w, void *y, void *residual_out,
                     int64_t rows, int64_t hidden, float eps, int dtype, const rmsnorm_plan_t *plan,
                     rmsnorm_stream_t stream) {
    Op o;
    int st = make_contig(x, residual, w, y, residual_out, rows, hidden, eps, 0.f, dtype, &o);
    if (st != RMSNORM_OK) return st;
    // fp32 I/O: the plain weight mode already rounds h * r to fp32 before the weight multiply.
    if (w != nullptr && dtype == RMSNORM_BF16) o.wm = rrn::kWeightCast;
    return run(o, plan, stream);
}

int rmsnorm_qk_fwd(const void *x, void *y, int64_t tokens, int64_t x_token_stride, int64_t y_token_stride,
                   int32_t q_heads, int32_t k_heads, int64_t head_dim, const void *q_w, const void *k_w,
                   float weight_bias, float eps, int dtype, const rmsnorm_plan_t *plan,
                   rmsnorm_stream_t stream) {
    Op o;
    int st = make_heads(x, y, tokens, x_token_stride, y_token_stride, q_heads, k_heads, head_dim, q_w, k_w,
                        weight_bias, eps, dtype, &o);
    if (st != RMSNORM_OK) return st;
    return run(o, plan, stream);
}

int rmsnorm_qk_plan_for(const void *x, const void *y, int64_t tokens, int64_t x_token_stride,
                        int64_t y_token_stride, int32_t q_heads, int32_t k_heads, int64_t head_dim,
                        const void *q_w, const void *k_w, int dtype, rmsnorm_plan_t *plan) {
    if (plan == nullptr) return RMSNORM_EINVAL;
    Op o;
    int st = make_heads(x, const_cast<void *>(y), tokens, x_token_stride, y_token_stride, q_heads, k_heads,
                        head_dim, q_w, k_w, 0.f, 0.f, dtype, &o);
    if (st != RMSNORM_OK) return st;
    if (!elem_aligned(o)) return RMSNORM_EINVAL;
    return plan_for_device(o, plan, nullptr);
}

int rmsnorm_tma_wait_test(const void *x, const void *residual, const void *w, void *y, void *residual_out,
                          int64_t rows, int64_t hidden, float eps, int dtype, const rmsnorm_plan_t *plan,
                          uint64_t wait_limit_ns, int withhold_release, rmsnorm_stream_t stream) {
    if (plan == nullptr || plan->kernel != RMSNORM_KERNEL_TMA) return RMSNORM_EINVAL;
    if (wait_limit_ns > kWaitLimitNs || (withhold_release != 0 && withhold_release != 1)) return RMSNORM_EINVAL;
    Op o;
    int st = make_contig(x, residual, w, y, residual_out, rows, hidden, eps, 0.f, dtype, &o);
    if (st != RMSNORM_OK) return st;
    o.wait_ns = wait_limit_ns == 0 ? kWaitLimitNs : wait_limit_ns;
    o.withhold = withhold_release;
    return run(o, plan, stream);
}

int64_t rmsnorm_max_hidden(int dtype) {
    return (dtype == RMSNORM_F32 || dtype == RMSNORM_BF16) ? kMaxHidden : 0;
}

int rmsnorm_reg_max_chunks(void) { return rrn::kRegMaxCH; }

int rmsnorm_wait_timeouts(uint32_t *count) {
    if (count == nullptr) return RMSNORM_EINVAL;
    unsigned int n = 0;
    if (rrn::tma_timeouts_read(&n) != 0) {
        (void)cudaGetLastError();
        return RMSNORM_ECUDA;
    }
    *count = n;
    return RMSNORM_OK;
}

const char *rmsnorm_strerror(int status) {
    switch (status) {
        case RMSNORM_OK: return "ok";
        case RMSNORM_EINVAL: return "invalid argument";
        case RMSNORM_EUNSUPPORTED: return "hidden size above the supported maximum";
        case RMSNORM_ECUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

const char *rmsnorm_build_info(void) {
    return "row_reduction_norm_gb300 fused RMSNorm / LayerNorm 0.3; target sm_103a; kernels: register (warp/"
           "CTA/persistent), shared-memory ring fed by bulk copies, two/three-pass; contiguous rows and Q/K head "
           "rows; weight, weight + bias, weight after a bf16 cast, no weight; MXFP8 / NVFP4 outputs";
}

}  // extern "C"
