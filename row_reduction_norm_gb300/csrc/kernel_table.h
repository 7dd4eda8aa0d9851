// kernel_table.h -- lookup of the compiled kernel instantiations (internal).
#pragma once

namespace rrn {

// Threads per row / chunk bounds compiled for the register kernel.
constexpr int kRegMaxGT = 512;        // contiguous rows
constexpr int kRegMaxGTHeads = 32;    // head rows (heads are short)
constexpr int kRegMaxCH = 8;
// Block sizes compiled for the two-pass kernel.
constexpr int kLoopBlocks[3] = {64, 256, 1024};

// dtype: 0 = f32, 1 = bf16; wm: 0 no weight, 1 weight, 2 weight + bias,
// 3 weight after a bf16 cast of the normalised value.
// Each returns the __global__ function as a launchable pointer, or nullptr
// when that combination is not compiled.
const void *reg_contig_f32_plain(int gt, int ch, int wm);
const void *reg_contig_f32_res(int gt, int ch, int wm);
const void *reg_contig_bf16_plain(int gt, int ch, int wm);
const void *reg_contig_bf16_res(int gt, int ch, int wm);
const void *reg_heads_f32(int gt, int ch, int wm);
const void *reg_heads_bf16(int gt, int ch, int wm);
const void *loop_contig(int dtype, int block, bool vec, bool res, int wm);
const void *loop_heads(int dtype, int block, bool vec, int wm);
// The cast-order weight mode (bf16 contiguous rows; the bulk-copy kernel's
// instantiations are in tma_kernel).
const void *reg_contig_bf16_cast(int gt, int ch, bool res);
const void *loop_contig_bf16_cast(int block, bool vec, bool res);

// RMSNorm with MXFP8 output (contiguous rows, register kernel only).
const void *mx_reg_f32_plain(int gt, int ch, int wm);
const void *mx_reg_f32_res(int gt, int ch, int wm);
const void *mx_reg_bf16_plain(int gt, int ch, int wm);
const void *mx_reg_bf16_res(int gt, int ch, int wm);

inline const void *mx_kernel(int dtype, int gt, int ch, bool res, int wm) {
    if (dtype == 1) return res ? mx_reg_bf16_res(gt, ch, wm) : mx_reg_bf16_plain(gt, ch, wm);
    return res ? mx_reg_f32_res(gt, ch, wm) : mx_reg_f32_plain(gt, ch, wm);
}

// RMSNorm with NVFP4 output (bf16 I/O, contiguous rows, register kernel only).
const void *nv_reg_bf16_plain(int gt, int ch, int wm);
const void *nv_reg_bf16_res(int gt, int ch, int wm);

inline const void *nv_kernel(int dtype, int gt, int ch, bool res, int wm) {
    if (dtype != 1) return nullptr;
    return res ? nv_reg_bf16_res(gt, ch, wm) : nv_reg_bf16_plain(gt, ch, wm);
}

// RMSNorm with the row staged in shared memory by bulk copies (contiguous
// rows, 16-byte units): 512 consumer threads and three producer warps a
// block; rings of pieces of 512 x 16 x pc bytes (pc: 1, 2 or 4) for x, the
// residual and the weight, kTmaMaxSlots slots in all, after the
// 2 x kTmaMaxSlots mbarriers.
constexpr int kTmaGT = 512;
constexpr int kTmaBlock = kTmaGT + 3 * 32;
constexpr int kTmaMaxSlots = 32;
constexpr int kTmaBarBytes = 2 * kTmaMaxSlots * 8;
constexpr int tma_piece_bytes(int pc) { return kTmaGT * 16 * pc; }
constexpr int tma_smem_bytes(int pc, int slots) { return kTmaBarBytes + slots * tma_piece_bytes(pc); }
// wg: the weight is read from global memory (no weight ring) rather than
// held resident in shared memory.
const void *tma_kernel(int dtype, int pc, bool res, int wm, bool wg);
// The same kernel with an MXFP8 (out 1: f32, bf16) or NVFP4 (out 2: bf16)
// output, 16 KB pieces (pc 2).
const void *tma_quant_kernel(int dtype, bool res, int wm, int out, bool wg);
// Reads the count of blocks whose bounded waits ran out (current device); 0 or -1.
int tma_timeouts_read(unsigned int *out);

// RMSNorm of contiguous rows with a residual, a row split over the blocks of
// a thread-block cluster: kClusterGT threads a block, each block a slice of
// kClusterGT * ch 16-byte units, up to kClusterMaxCtas blocks a cluster.
// Compiled for ch 4 and 5 (bf16, fp32) and 8 (fp32), with a residual only.
constexpr int kClusterGT = 256;
constexpr int kClusterMaxCtas = 8;
const void *cluster_kernel(int dtype, int ch, bool res, int wm);

// LayerNorm (contiguous rows); aff: 0 none, 1 weight, 2 weight and bias.
constexpr int kLnMaxGT = 256;
const void *ln_reg_f32(int gt, int ch, bool res, int aff);
const void *ln_reg_bf16(int gt, int ch, bool res, int aff);
const void *ln_loop(int dtype, int block, bool vec, bool res, int aff);

inline const void *reg_kernel(int dtype, int gt, int ch, bool res, int wm, bool heads) {
    if (heads) return res ? nullptr : (dtype == 1 ? reg_heads_bf16(gt, ch, wm) : reg_heads_f32(gt, ch, wm));
    if (dtype == 1) return res ? reg_contig_bf16_res(gt, ch, wm) : reg_contig_bf16_plain(gt, ch, wm);
    return res ? reg_contig_f32_res(gt, ch, wm) : reg_contig_f32_plain(gt, ch, wm);
}

inline const void *loop_kernel(int dtype, int block, bool vec, bool res, int wm, bool heads) {
    if (heads) return res ? nullptr : loop_heads(dtype, block, vec, wm);
    return loop_contig(dtype, block, vec, res, wm);
}

}  // namespace rrn
