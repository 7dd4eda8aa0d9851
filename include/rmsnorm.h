/*
 * rmsnorm.h -- C ABI of the GB300 (sm_103a) fused row-wise RMSNorm library
 * (with its LayerNorm and fused Q+K head-norm variants).
 *
 * The operation (one row at a time, rows of a row-major [rows, hidden] tensor):
 *
 *   h_i          = x_i,   or  h_i = RN_T(x_i + residual_i) with a residual
 *   residual_out = h                                   (only with a residual)
 *   y_i          = RN_T( h_i * rsqrt(mean_j(h_j^2) + eps) * w_i )
 *                  (w_i dropped when no weight is given)
 *
 * Definition: "Building a GPU compiler from scratch: from PyTorch to CUDA via
 * multi-level IR (Emmy)" -- the running example (mean of the squares of the
 * row, plus epsilon, inverse square root, times each element and its learned
 * weight) and section "Tensor IR" (square, sum, division by the count, plus
 * epsilon, rsqrt, two multiplications).  The weight / no-weight and per-dtype
 * specialisation follows "CuTeDSL at Perplexity", section on the large
 * configuration space.  RN_T is round-to-nearest-even to the I/O type T.
 * The residual add is not described on the pages; the reading taken is that
 * residual_out is the sum rounded once to T and the norm is taken of it.
 *
 * Arithmetic: inputs are widened to fp32; the sum of squares is formed in
 * fp32 in a fixed order that depends only on (hidden, dtype, alignment, and,
 * for rows longer than 32 KB, whether a residual is given), so every call
 * gives bit-identical results for a row, whatever the row count, grid or
 * stream ("batch invariant").  Accuracy: y is within 1 ulp of the
 * correctly rounded result for bf16 and within 2e-6 relative for fp32;
 * residual_out is the correctly rounded sum (bit-exact).
 *
 * Conventions common to every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, on the
 *    caller's current CUDA device; the library allocates and frees nothing.
 *    (rmsnorm_fwd_host takes HOST tensors and a caller-owned device
 *    workspace; it allocates no memory either.)
 *  - Every tensor shares one I/O type (dtype).  x, residual, y and
 *    residual_out are contiguous row-major [rows, hidden]; w is [hidden].
 *  - Calls are asynchronous on `stream` (0 = the legacy default stream) and
 *    never synchronise.  Errors detected before the launch return a status
 *    and launch nothing.
 *  - Aliasing: an input may be the very same buffer as an output (y == x,
 *    residual_out == residual, ...): each thread reads its elements before it
 *    writes them.  y and residual_out must not overlap each other, w must not
 *    overlap an output, and partial overlaps are undefined.
 *  - Alignment: when every pointer is 16-byte aligned and hidden * sizeof(T)
 *    is a multiple of 16, rows move with 128-bit loads and stores; otherwise a
 *    scalar path runs (same results up to the stated tolerance).
 *  - Thread safety: entry points may be called from several host threads.
 *    The library's state is a per-device cache of the SM count and of
 *    kernel occupancy, and the three streams and seven events per device
 *    that rmsnorm_fwd_host creates at its first call there.
 */
#ifndef ROW_REDUCTION_NORM_GB300_RMSNORM_H
#define ROW_REDUCTION_NORM_GB300_RMSNORM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *rmsnorm_stream_t;

/* I/O types (the `dtype` argument). */
enum { RMSNORM_F32 = 0, RMSNORM_BF16 = 1 };

/* Status codes. */
enum {
    RMSNORM_OK = 0,
    RMSNORM_EINVAL = -1,        /* null x or y, rows < 0, hidden <= 0, unknown dtype,
                                   eps negative or not finite, residual given without
                                   residual_out or the reverse, bad plan            */
    RMSNORM_EUNSUPPORTED = -2,  /* hidden above rmsnorm_max_hidden()               */
    RMSNORM_ECUDA = -3          /* the CUDA runtime reported an error (launch,
                                   device query)                                    */
};

/* Kernel families (rmsnorm_plan_t.kernel). */
enum {
    RMSNORM_KERNEL_REG = 0,   /* row held in registers, 128-bit I/O, one pass     */
    RMSNORM_KERNEL_LOOP = 1,  /* row streamed twice (second read from L2): any
                                 alignment; planned for unaligned rows and for
                                 rows past 192 KB without a residual           */
    RMSNORM_KERNEL_TMA = 2,   /* row staged in shared memory by bulk (TMA) copies:
                                 rings for x, residual and weight fed by three
                                 producer warps, 512 threads a row; contiguous
                                 RMSNorm rows past 32 KB without a residual
                                 (and block-scaled outputs of rows too long for
                                 registers)                                     */
    RMSNORM_KERNEL_CLUSTER = 3 /* row split over the 2..8 blocks of a thread-block
                                 cluster, each holding a slice in registers; the
                                 blocks' partial sums meet in distributed shared
                                 memory behind one cluster barrier; contiguous
                                 RMSNorm rows past 32 KB with a residual       */
};

/* Regimes (rmsnorm_plan_t.regime), a summary of how rows map to threads. */
enum {
    RMSNORM_REGIME_WARP = 0,        /* 4..32 lanes of one warp per row               */
    RMSNORM_REGIME_CTA = 1,         /* several warps per row, shared-memory combine  */
    RMSNORM_REGIME_PERSISTENT = 2,  /* grid capped at the resident capacity; blocks
                                       stride over the rows                          */
    RMSNORM_REGIME_LOOPED = 3,      /* RMSNORM_KERNEL_LOOP                           */
    RMSNORM_REGIME_SMEM = 4,        /* RMSNORM_KERNEL_TMA: one block per SM, blocks
                                       stride over the rows                          */
    RMSNORM_REGIME_CLUSTER = 5      /* RMSNORM_KERNEL_CLUSTER: one cluster a row     */
};

/*
 * A launch plan.  The per-row schedule (kernel, threads_per_row, vec_elems,
 * block_threads, cluster_ctas) depends only on hidden, dtype and the
 * alignment of the pointers (and, for rows longer than 32 KB, on whether a
 * residual is given);
 * rows sizes the grid, may pick a chunk count that fits the row exactly and
 * may give each row a block of its own (rows_per_block 1), none of which ever
 * changes a result (chunks past the row end add exact zeros; which block takes
 * a row does not matter).
 */
typedef struct {
    int32_t kernel;             /* RMSNORM_KERNEL_*                                   */
    int32_t regime;             /* RMSNORM_REGIME_*                                   */
    int32_t threads_per_row;    /* REG: 4..512 (4..32 for head rows), power of two;
                                   LOOP: block_threads; TMA: 512; CLUSTER: 256 *
                                   cluster_ctas                                       */
    int32_t chunks_per_thread;  /* REG: vector chunks per thread (an upper bound:
                                   slots past the row end stay idle); 1, 2, 4 or 8,
                                   and 3 or 6 for contiguous RMSNorm / LayerNorm rows
                                   in the I/O type (planning takes them for LayerNorm,
                                   for RMSNorm rows of a warp or less, and for wider
                                   RMSNorm rows in launches of more than one wave of
                                   blocks); LOOP: 0; TMA: chunks per thread
                                   in one ring piece: 1, 2 or 4 (8, 16 or 32 KB
                                   pieces; 28, 14 or 7 slots of shared memory, of
                                   which avail / 7 (at least 1) go to a streamed
                                   residual ring; a weight ring gets one slot per
                                   piece (the weight resident) when that leaves x
                                   a row and two spare slots, else there is none
                                   and the weight is read from global memory; the
                                   rest, which must hold a whole row, goes to x);
                                   CLUSTER: chunks per thread of a block's slice of
                                   256 * chunks_per_thread chunks: 4 (16 KB), 5
                                   (20 KB; planned for rows of 64 to 80 KB), or 8
                                   (32 KB, fp32 only; planned for rows past 128 KB),
                                   a result depending on it (not on cluster_ctas)  */
    int32_t vec_elems;          /* elements per load: 16 / sizeof(T), or 1 (scalar)  */
    int32_t block_threads;      /* threads per block: REG max(threads_per_row, 256),
                                   or max(threads_per_row, 128) for LayerNorm;
                                   LOOP: threads_per_row; TMA: 608; CLUSTER: 256      */
    int32_t rows_per_block;     /* rows one block handles per loop iteration: REG
                                   block_threads / threads_per_row, or (RMSNorm only)
                                   fewer, down to 1; planning takes one warp of rows
                                   a block (1 for rows of 32 threads or more) when
                                   that needs no more blocks than the device has
                                   SMs (decode batches); other kernels 1           */
    int32_t persistent;         /* 1 if grid < row blocks (blocks stride over rows)   */
    int32_t pdl;                /* 1: launch with programmatic stream serialisation
                                   (the kernel may start while the previous kernel on
                                   the stream drains; it reads no input before that
                                   kernel has completed).  Planning sets 1.          */
    int32_t cluster_ctas;       /* CLUSTER: blocks of a cluster, which share a row,
                                   2..8, covering the row (the fewest that do, in
                                   planning); 0 for the other kernels              */
    int64_t grid;               /* blocks launched (0 when rows == 0); CLUSTER: a
                                   multiple of cluster_ctas (rows * cluster_ctas
                                   in planning; fewer clusters stride over rows)   */
} rmsnorm_plan_t;

/*
 * Fused RMSNorm forward (the op above).
 *   x            [rows, hidden]  input
 *   residual     [rows, hidden]  optional (NULL): added to x before the norm
 *   w            [hidden]        optional (NULL): per-element weight
 *   y            [rows, hidden]  output
 *   residual_out [rows, hidden]  required iff residual is given: receives h
 *   rows >= 0 (0 is a successful no-op that reads no pointer, which may then
 *   be NULL), 1 <= hidden <= rmsnorm_max_hidden(dtype)
 *   eps          finite, >= 0; used as the float value passed
 *   dtype        RMSNORM_F32 or RMSNORM_BF16
 * Returns RMSNORM_OK or a negative status (see above).
 */
int rmsnorm_fwd(const void *x, const void *residual, const void *w, void *y,
                void *residual_out, int64_t rows, int64_t hidden, float eps,
                int dtype, rmsnorm_stream_t stream);

/*
 * Regime dispatch ("CuTeDSL at Perplexity", section on prefill and decode
 * specialisation: the grid and block shape of a row kernel follow the token
 * count, the hidden size, the data type and the device's SM count).  The
 * plan calls below expose that choice; rmsnorm_regime names the regime alone.
 *
 * rmsnorm_regime: the RMSNORM_REGIME_* that rmsnorm_fwd runs on the current
 * device for `rows` rows of `hidden` elements of `dtype`, with 16-byte
 * aligned tensors, a weight and no residual (rmsnorm_plan_for answers for
 * any other pointers).  rows >= 0 and hidden, dtype as for rmsnorm_fwd.
 * Queries the SM count and the kernel's occupancy once per device.  Returns
 * the regime (>= 0) or a negative status: RMSNORM_EINVAL,
 * RMSNORM_EUNSUPPORTED, or RMSNORM_ECUDA (no usable device).
 */
int rmsnorm_regime(int64_t rows, int64_t hidden, int dtype);

/*
 * Pure host planning (no CUDA call): the plan rmsnorm_fwd would use without
 * a residual on a device with `sm_count` SMs where the chosen kernel keeps
 * `blocks_per_sm` blocks resident (with a residual, rows longer than 32 KB
 * take RMSNORM_KERNEL_CLUSTER instead: 16 KB slices up to 128 KB rows, but
 * 20 KB for rows of 64 to 80 KB, and 32 KB slices past 128 KB).  vec_ok: 1 if every pointer is 16-byte aligned and
 * hidden * sizeof(T) is a multiple of 16.  Returns a status.
 */
int rmsnorm_plan(int64_t rows, int64_t hidden, int dtype, int vec_ok, int sm_count,
                 int blocks_per_sm, rmsnorm_plan_t *plan);

/*
 * rmsnorm_plan with the residual stated: has_residual 1 gives the plan
 * rmsnorm_fwd uses when a residual (and residual_out) is passed, 0 is
 * rmsnorm_plan.  Pure host planning, no CUDA call.  Returns a status
 * (RMSNORM_EINVAL for has_residual other than 0 or 1).
 */
int rmsnorm_plan_ex(int64_t rows, int64_t hidden, int dtype, int vec_ok, int has_residual,
                    int sm_count, int blocks_per_sm, rmsnorm_plan_t *plan);

/*
 * The plan rmsnorm_fwd would use for these pointers on the current device
 * (queries the SM count and the kernel's occupancy once per device).
 */
int rmsnorm_plan_for(const void *x, const void *residual, const void *w, const void *y,
                     const void *residual_out, int64_t rows, int64_t hidden, int dtype,
                     rmsnorm_plan_t *plan);

/*
 * rmsnorm_fwd with a caller-chosen plan (tests and schedule sweeps).  The plan
 * is validated against the shape and the pointers: a REG plan must cover the
 * row (threads_per_row * chunks_per_thread * vec_elems >= hidden, with a
 * compiled chunks_per_thread, see rmsnorm_plan_t), block_threads and
 * rows_per_block must match threads_per_row, a TMA plan must fit the row in
 * its ring (see rmsnorm_plan_t), a CLUSTER plan needs a residual, a compiled
 * chunks_per_thread, 2..8 cluster_ctas that cover the row and a grid that is
 * a multiple of cluster_ctas, a vector plan (REG, TMA, CLUSTER) needs aligned
 * pointers, grid >= 1, pdl 0 or 1 and cluster_ctas 0 for the other kernels.
 * Returns RMSNORM_EINVAL for a plan that does not fit.
 */
int rmsnorm_fwd_plan(const void *x, const void *residual, const void *w, void *y,
                     void *residual_out, int64_t rows, int64_t hidden, float eps,
                     int dtype, const rmsnorm_plan_t *plan, rmsnorm_stream_t stream);

/*
 * rmsnorm_fwd with a weight bias and an optional plan:
 *   y_i = RN_T( h_i * rsqrt(mean(h^2) + eps) * (w_i + weight_bias) )
 * The constant added to every weight element is the "weight bias" knob of
 * "CuTeDSL at Perplexity" (configuration-space section; WEIGHT_BIAS in
 * section "QK Norm"), read as an offset of the weight: weight_bias = 1 gives
 * the (1 + w) form.  weight_bias = 0 is exactly rmsnorm_fwd.  A non-zero
 * weight_bias requires w; it must be finite.  plan may be NULL (the library's
 * plan) or a plan as for rmsnorm_fwd_plan.  Other arguments, layout and
 * status codes as rmsnorm_fwd.
 */
int rmsnorm_fwd_ex(const void *x, const void *residual, const void *w, void *y,
                   void *residual_out, int64_t rows, int64_t hidden, float eps,
                   float weight_bias, int dtype, const rmsnorm_plan_t *plan,
                   rmsnorm_stream_t stream);

/*
 * rmsnorm_fwd in the op-by-op cast order of an eager framework
 * ("model-as-a-kernel", sections "Method" and "Correctness": eager bf16
 * semantics op for op, its fused rmsnorm bitwise).  The card does not spell
 * the order out; the reading taken is a norm whose weight multiply is an op of
 * its own:
 *   n_i = RN_T( h_i * rsqrt(mean(h^2) + eps) )      (statistics in fp32)
 *   y_i = RN_T( n_i * w_i )                         (n_i without a weight)
 * For bf16 this differs from rmsnorm_fwd, which rounds once; for fp32 I/O the
 * two calls run the same arithmetic.  Without a weight it is rmsnorm_fwd.
 * Accuracy (bf16): n_i is the correctly rounded normalised value except where
 * the exact value lies within 2e-6 (relative) of a bf16 rounding midpoint,
 * where it may be the other neighbour; y_i is then exactly RN_T(n_i * w_i).
 * plan may be NULL (the library's plan) or a plan as for rmsnorm_fwd_plan;
 * rmsnorm_plan_for returns the plan this call uses.  Other arguments, layout,
 * ownership and status codes as rmsnorm_fwd.
 */
int rmsnorm_fwd_cast(const void *x, const void *residual, const void *w, void *y,
                     void *residual_out, int64_t rows, int64_t hidden, float eps,
                     int dtype, const rmsnorm_plan_t *plan, rmsnorm_stream_t stream);

/*
 * Fused query + key per-head RMSNorm in one launch ("CuTeDSL at Perplexity",
 * section "QK Norm": per-head norm over 64..256 elements, the kernel picks
 * the query or key weight per head; the model-as-a-kernel card lists the
 * Qwen3-style qk RMSNorm).  Every head is one row of head_dim elements,
 * normalised on its own with the op of rmsnorm_fwd_ex (no residual).
 *
 * Layout (element offsets; token rows of a packed projection such as
 * [tokens, (q_heads + k_heads + v_heads) * head_dim]):
 *   query head j of token t:  t * x_token_stride + j * head_dim
 *   key head j of token t:    t * x_token_stride + (q_heads + j) * head_dim
 * y uses the same layout with y_token_stride.  Elements of a token row past
 * (q_heads + k_heads) * head_dim (the value heads) are neither read nor
 * written.  y == x (same stride) normalises in place.
 *   q_w, k_w    [head_dim] weights of the query and key heads: both or neither
 *   weight_bias as rmsnorm_fwd_ex (requires weights when non-zero)
 *   tokens >= 0 (0: no-op); q_heads, k_heads >= 0 with q_heads + k_heads >= 1;
 *   1 <= head_dim <= rmsnorm_max_hidden(dtype);
 *   x_token_stride, y_token_stride >= (q_heads + k_heads) * head_dim
 *   plan        NULL (the library's plan) or a caller plan (validated)
 * Returns RMSNORM_OK or a negative status (RMSNORM_EINVAL also for strides
 * shorter than the heads, or y == x with different strides).
 */
int rmsnorm_qk_fwd(const void *x, void *y, int64_t tokens, int64_t x_token_stride,
                   int64_t y_token_stride, int32_t q_heads, int32_t k_heads,
                   int64_t head_dim, const void *q_w, const void *k_w, float weight_bias,
                   float eps, int dtype, const rmsnorm_plan_t *plan,
                   rmsnorm_stream_t stream);

/* The plan rmsnorm_qk_fwd would use for these arguments on the current device. */
int rmsnorm_qk_plan_for(const void *x, const void *y, int64_t tokens, int64_t x_token_stride,
                        int64_t y_token_stride, int32_t q_heads, int32_t k_heads,
                        int64_t head_dim, const void *q_w, const void *k_w, int dtype,
                        rmsnorm_plan_t *plan);

/*
 * RMSNorm with a block-scaled MXFP8 output (OCP Microscaling Formats v1.0:
 * E4M3 elements, one E8M0 scale per 32 elements; block-scaled low-precision
 * formats are named in "CuTeDSL at Perplexity", section "Blackwell
 * support").  The op's fp32 values v_i = h_i * r * (w_i + weight_bias) (as
 * rmsnorm_fwd_ex, before any rounding to the I/O type) are quantised in
 * blocks of 32 consecutive elements of a row:
 *   s       = floor(log2(max |v|)) - 8, clamped to [-127, 127] (-127 for a zero block)
 *   scales  [rows, hidden / 32] bytes: E8M0 code s + 127
 *   codes   [rows, hidden] bytes: E4M3 of v_i / 2^s, nearest-even, saturated at 448
 * A block holding NaN or Inf is a NaN block (scale 0xFF, every code 0x7F).
 * hidden must be a multiple of 32 and x, residual, w, codes and
 * residual_out 16-byte aligned (else RMSNORM_EINVAL).  Rows past 32768 bf16
 * or 16384 fp32 elements run on RMSNORM_KERNEL_TMA (16 KB pieces) while its
 * rings hold them: every bf16 width, fp32 up to 40960 elements with a
 * residual and a weight (49152 with one of them, 57344 with neither), else
 * RMSNORM_EUNSUPPORTED.  residual_out
 * (required with a residual) receives h in the I/O type.  A code chosen by
 * the kernel may differ from the correctly rounded one only when the exact
 * value lies within the fp32 error of the op (about 1e-6 relative) of an
 * E4M3 rounding midpoint, and likewise a scale when the block's maximum lies
 * that close to a power of two.
 */
int rmsnorm_fwd_mxfp8(const void *x, const void *residual, const void *w, void *codes,
                      void *scales, void *residual_out, int64_t rows, int64_t hidden,
                      float eps, float weight_bias, int dtype, const rmsnorm_plan_t *plan,
                      rmsnorm_stream_t stream);

/* The plan rmsnorm_fwd_mxfp8 would use for these pointers on the current device. */
int rmsnorm_mxfp8_plan_for(const void *x, const void *residual, const void *w,
                           const void *codes, const void *scales, const void *residual_out,
                           int64_t rows, int64_t hidden, int dtype, rmsnorm_plan_t *plan);

/*
 * RMSNorm with a block-scaled NVFP4 output: E2M1 elements (magnitudes 0, 0.5,
 * 1, 1.5, 2, 3, 4, 6), one E4M3 scale per 16 elements and a per-tensor fp32
 * scale S given by the caller ("CuTeDSL at Perplexity", section "Blackwell
 * support", names NVFP4 without a recipe; the reading taken is that a value
 * decodes as code * scale * S).  For each block of 16 consecutive elements of
 * a row, with the op's fp32 values v_i as for rmsnorm_fwd_mxfp8:
 *   scales  [rows, hidden / 16] bytes: E4M3(amax / (6 S)), nearest-even, saturating
 *   codes   [rows, hidden / 2] bytes: E2M1(v_i / (scale * S)), nearest-even,
 *           saturated at 6, two a byte, element 2k in the low nibble
 *           (all 0 when the block's scale is 0)
 * A block holding NaN or Inf gets the E4M3 NaN 0x7F as its scale and codes 0.
 * bf16 I/O only (fp32: RMSNORM_EUNSUPPORTED); hidden a multiple of 16;
 * tensor_scale > 0 and finite; x, residual, w, codes, residual_out 16-byte
 * aligned.  Rows past 32768 elements run on RMSNORM_KERNEL_TMA (16 KB
 * pieces).  Codes and scales may differ from the correctly rounded ones only
 * where the exact value lies within the op's fp32 error of a rounding
 * boundary, as for MXFP8.
 */
int rmsnorm_fwd_nvfp4(const void *x, const void *residual, const void *w, void *codes,
                      void *scales, void *residual_out, int64_t rows, int64_t hidden,
                      float eps, float weight_bias, float tensor_scale, int dtype,
                      const rmsnorm_plan_t *plan, rmsnorm_stream_t stream);

/* The plan rmsnorm_fwd_nvfp4 would use for these pointers on the current device. */
int rmsnorm_nvfp4_plan_for(const void *x, const void *residual, const void *w,
                           const void *codes, const void *scales, const void *residual_out,
                           int64_t rows, int64_t hidden, int dtype, rmsnorm_plan_t *plan);

/*
 * Fused row-wise LayerNorm ("GPT-2 on the GPU", section "The Whole Model as
 * One Kernel": mean, variance, (x - mean) / sqrt(var + eps), weight times the
 * normalised value plus bias):
 *   h    = x, or RN_T(x + residual) written to residual_out
 *   mu   = mean(h),  var = mean((h - mu)^2)   (population variance)
 *   y_i  = RN_T( (h_i - mu) * rsqrt(var + eps) * w_i + b_i )
 * w and b are optional [hidden] tensors (b requires w); without w the
 * normalised value is returned.  Layout, aliasing, alignment, plan and
 * status codes as rmsnorm_fwd_ex (REG plans up to 256 threads per row).
 * The statistics are formed in fp32 in a fixed order; the variance is taken
 * of the centred values (a second pass over the row held on chip).
 */
int layernorm_fwd(const void *x, const void *residual, const void *w, const void *b, void *y,
                  void *residual_out, int64_t rows, int64_t hidden, float eps, int dtype,
                  const rmsnorm_plan_t *plan, rmsnorm_stream_t stream);

/* The plan layernorm_fwd would use for these pointers on the current device. */
int layernorm_plan_for(const void *x, const void *residual, const void *w, const void *b,
                       const void *y, const void *residual_out, int64_t rows, int64_t hidden,
                       int dtype, rmsnorm_plan_t *plan);

/*
 * The op of rmsnorm_fwd (Emmy page, running example and section "Tensor
 * IR") on rows that live in HOST memory: x, residual, w, y and residual_out
 * are host pointers, with rmsnorm_fwd's layout and argument rules.  The rows
 * go through the current device in chunks of chunk_rows rows (the last may
 * be shorter): a chunk's inputs are copied into one of the two halves of
 * `workspace`, one rmsnorm_fwd launch normalises them there, and its outputs
 * are copied back; uploads, launches and read-backs run on three streams of
 * the library's, so a chunk's uploads overlap the previous chunk's launch
 * and read-backs and both copy directions run at once.  The pages describe
 * no such call: it is the op end to end from host memory, the form a caller
 * holding activations in host memory uses (and the benchmark's end-to-end
 * figure).
 *   workspace        DEVICE memory owned by the caller, 256-byte aligned,
 *                    workspace_bytes >= rmsnorm_host_workspace_bytes(
 *                    chunk_rows, hidden, dtype, residual != NULL); used by
 *                    no one else until the call's work on `stream` is done
 *   chunk_rows       >= 1
 *   stream           the call's copies start after the work issued on
 *                    `stream` before the call, and work issued on `stream`
 *                    after it starts after the call's last read-back:
 *                    synchronise `stream` before reading y on the host
 * Overlap needs page-locked host memory (cudaHostAlloc, cudaHostRegister);
 * with pageable memory the results are the same and the CUDA runtime
 * serialises the copies.  Each chunk is one rmsnorm_fwd launch on 256-byte
 * aligned device copies, so the results are those of rmsnorm_fwd on such
 * copies of the same rows, bit for bit (the schedule does not depend on the
 * row count).  Calls on one device are queued one at a time (a per-device
 * lock held while the copies and launches are issued, not while they run);
 * not for use while a stream is being captured.  Returns RMSNORM_OK or a
 * negative status: RMSNORM_EINVAL for a NULL x or y with rows > 0, a
 * residual without residual_out or the reverse, chunk_rows < 1, a NULL,
 * misaligned or too small workspace, or rmsnorm_fwd's own argument errors;
 * RMSNORM_EUNSUPPORTED; RMSNORM_ECUDA.  rows == 0 does nothing.
 */
int rmsnorm_fwd_host(const void *x, const void *residual, const void *w, void *y,
                     void *residual_out, int64_t rows, int64_t hidden, float eps, int dtype,
                     void *workspace, uint64_t workspace_bytes, int64_t chunk_rows,
                     rmsnorm_stream_t stream);

/*
 * Device workspace bytes rmsnorm_fwd_host needs: the weight, then two halves
 * of chunk_rows rows of x and y (and of residual and residual_out with
 * has_residual = 1), each part starting on a 256-byte boundary.  Returns the
 * byte count (> 0) or a negative status (RMSNORM_EINVAL: chunk_rows < 1,
 * hidden < 1, unknown dtype, has_residual not 0 or 1, a size that overflows;
 * RMSNORM_EUNSUPPORTED: hidden above rmsnorm_max_hidden).
 */
int64_t rmsnorm_host_workspace_bytes(int64_t chunk_rows, int64_t hidden, int dtype, int has_residual);

/*
 * The op of rmsnorm_fwd (Emmy page, running example and section "Tensor
 * IR") on host rows, as rmsnorm_fwd_host computes it, without a workspace
 * argument: the library's own 64 MiB of device scratch (a file-scope
 * __device__ array, one per device, its address taken with
 * cudaGetSymbolAddress at the first call) serves as the workspace, with
 * chunks of as many rows as fit it.  The call allocates
 * nothing; the scratch belongs to the library's device image (with lazy
 * module loading, claimed on the device at the first call).  Arguments,
 * ordering on `stream`, results (bit for bit) and statuses as
 * rmsnorm_fwd_host; calls on one device share the scratch and are ordered
 * by that call's per-device pipeline.
 */
int rmsnorm_fwd_host_static(const void *x, const void *residual, const void *w, void *y,
                            void *residual_out, int64_t rows, int64_t hidden, float eps, int dtype,
                            rmsnorm_stream_t stream);

/* Largest supported hidden size for a dtype (0 for an unknown dtype). */
int64_t rmsnorm_max_hidden(int dtype);

/* Largest chunks_per_thread a REG plan may use. */
int rmsnorm_reg_max_chunks(void);

/*
 * Every wait inside the RMSNORM_KERNEL_TMA kernel (for a bulk copy to land,
 * for a ring slot to be released) gives up after one second; the block then
 * finishes its rows without waiting (its outputs are not valid), waits, again
 * at most a second each, for its copies still in flight, and adds 1 to a
 * per-device counter.  A consumer warp that gave up releases no ring slot from
 * then on, so no copy is ever started into a slot whose previous copy may
 * still be landing.  The launch itself returned RMSNORM_OK when it was
 * issued; this counter is how the host learns that a block gave up.  This
 * reads that counter for the current device (the count since the library was
 * loaded; 0 unless a launch went wrong).  It is a blocking device-to-host
 * read: call it after synchronising the streams that ran the kernels, and
 * not while a stream is being captured.
 * Returns RMSNORM_OK, RMSNORM_EINVAL (count NULL) or RMSNORM_ECUDA.
 */
int rmsnorm_wait_timeouts(uint32_t *count);

/*
 * Test hook of the bounded waits above (the pages describe no such hook):
 * rmsnorm_fwd_plan with a RMSNORM_KERNEL_TMA plan (else RMSNORM_EINVAL),
 * every wait of the kernel limited to wait_limit_ns nanoseconds (0: the
 * one-second default; at most one second), and, with withhold_release = 1,
 * one release of an x slot withheld by the first consumer warp of block 0.
 * That block's x producer then waits for a slot that never frees: its wait
 * runs out, so do the consumers' waits for the pieces it no longer copies,
 * the block finishes with no valid output for its rows, waits for its copies
 * in flight, and adds 1 to the count rmsnorm_wait_timeouts reads.  Blocks
 * other than block 0 and every launch with withhold_release = 0 compute the
 * op as rmsnorm_fwd_plan does.  Nothing faults and no wait is unbounded:
 * a test uses it to see the failure path work and the next launch succeed.
 * The launch is asynchronous like every other: its status says whether it
 * was launched, the counter whether a block gave up.
 */
int rmsnorm_tma_wait_test(const void *x, const void *residual, const void *w, void *y,
                          void *residual_out, int64_t rows, int64_t hidden, float eps, int dtype,
                          const rmsnorm_plan_t *plan, uint64_t wait_limit_ns, int withhold_release,
                          rmsnorm_stream_t stream);

/* Static text for a status code. */
const char *rmsnorm_strerror(int status);

/* Static text describing the build (target architecture, version). */
const char *rmsnorm_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* ROW_REDUCTION_NORM_GB300_RMSNORM_H */
