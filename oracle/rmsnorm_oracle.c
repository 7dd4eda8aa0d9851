/*
 * rmsnorm_oracle.c -- plain fp64 CPU reference for the fused row-wise RMSNorm.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline / reference legs load this file.  It shares
 * no code, header, table or helper with the CUDA library, and it does not
 * include anything from it.
 *
 * What it computes, for each row of a row-major [rows, hidden] tensor:
 *
 *   h_i   = x_i                               (no residual)
 *   h_i   = RN_T(x_i + residual_i)            (fused residual add; h is stored
 *                                               as residual_out, and the norm
 *                                               is taken of this rounded h)
 *   S     = sum_i h_i^2                        (fp64, index order)
 *   r     = 1 / sqrt(S / hidden + eps)
 *   y_i   = RN_T(h_i * r * w_i)                (w_i dropped with no weight)
 *   y_i   = RN_T(h_i * r * (w_i + b))          (weight bias b, when non-zero)
 *
 * Sources:
 *  - "Building a GPU compiler from scratch: from PyTorch to CUDA via
 *    multi-level IR (Emmy)", opening description of the running example: the
 *    mean of the squares of the row, plus epsilon, inverse square root, and a
 *    scale of every element by that value and by its learned weight.
 *  - Same page, section "Tensor IR": the step list square, sum, division by
 *    the count, addition of epsilon, rsqrt, two multiplications.  The loop
 *    below takes exactly those steps in that order.
 *  - The fused residual add, the optional weight and the bf16/fp32 I/O are
 *    not described on the pages; the reading taken is: h is the sum rounded
 *    once to the I/O type, and the norm is taken of that rounded h.
 *  - eps arrives as a float; its exact float value is used.
 *  - The weight bias is the "weight bias" knob of "CuTeDSL at Perplexity"
 *    (configuration-space section, WEIGHT_BIAS in section "QK Norm"), read as
 *    a constant added to every weight element (1 gives the (1 + w) form).
 *
 * Arithmetic: every step in IEEE binary64 with round-to-nearest-even, no
 * fused multiply-add (built with -ffp-contract=off) and no fast-math.  The
 * only rounding to the I/O type is the final one per output (and the one that
 * defines h with a residual).
 *
 * bf16 is the upper 16 bits of an IEEE binary32 value: 1 sign bit, 8 exponent
 * bits, 7 fraction bits.  It is decoded by placing the 16 bits on top of 16
 * zero bits.  Rounding a double to bf16 is done from that definition: round
 * the magnitude to 8 significant bits (a fixed quantum of 2^-133 below the
 * smallest normal 2^-126), ties to even, and overflow to infinity beyond the
 * largest finite value 255 * 2^120.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static uint16_t double_to_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);            /* a lies in [2^(e-1), 2^e)                  */
    int q = e - 8;           /* 8 significant bits: quantum 2^(e-1-7)      */
    if (q < -133)
        q = -133;            /* subnormal range: fixed quantum 2^-133      */
    double n = nearbyint(ldexp(a, -q));  /* exact scaling, ties to even    */
    double r = ldexp(n, q);
    if (r > ldexp(255.0, 120))           /* above the largest finite bf16  */
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)r;                  /* exact: r has <= 8 bits         */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

static double load_elem(const void *p, int64_t i, int dtype)
{
    if (dtype == ORACLE_BF16)
        return bf16_to_double(((const uint16_t *)p)[i]);
    return (double)((const float *)p)[i];
}

/* Round v to the I/O type and store it. */
static void store_elem(void *p, int64_t i, int dtype, double v)
{
    if (dtype == ORACLE_BF16)
        ((uint16_t *)p)[i] = double_to_bf16(v);
    else
        ((float *)p)[i] = (float)v;   /* C conversion: round to nearest even */
}

/* The value the I/O type holds for v (v rounded once to the type). */
static double round_to_type(double v, int dtype)
{
    if (dtype == ORACLE_BF16)
        return bf16_to_double(double_to_bf16(v));
    return (double)(float)v;
}

/* h_i: the row element that is normalised. */
static double row_input(const void *x, const void *residual, int64_t i, int dtype)
{
    double xi = load_elem(x, i, dtype);
    if (residual == NULL)
        return xi;
    return round_to_type(xi + load_elem(residual, i, dtype), dtype);
}

/*
 * The op's fp64 values v_i (y_i before its rounding to the I/O type) for one
 * row, and h written to residual_out when a residual is given.
 */
static void rms_row_values(const void *x, const void *residual, const void *w, int64_t row,
                           int64_t hidden, double e, double b, int dtype, double *v,
                           void *residual_out)
{
    const int64_t base = row * hidden;

    /* square and sum */
    double sum_sq = 0.0;
    for (int64_t i = 0; i < hidden; ++i) {
        double h = row_input(x, residual, base + i, dtype);
        sum_sq += h * h;
    }
    /* divide by the count, add epsilon, inverse square root */
    double mean_sq = sum_sq / (double)hidden;
    double inv_rms = 1.0 / sqrt(mean_sq + e);

    /* two multiplications */
    for (int64_t i = 0; i < hidden; ++i) {
        double h = row_input(x, residual, base + i, dtype);
        double t = h * inv_rms;
        if (w != NULL)
            t = t * (load_elem(w, i, dtype) + b);
        v[i] = t;
        if (residual_out != NULL)
            store_elem(residual_out, base + i, dtype, h);
    }
}

/*
 * Rows [row_begin, row_end) of the op.
 *   x, residual, w : inputs in the I/O type (residual and w may be NULL)
 *   y              : output in the I/O type
 *   y_exact        : optional fp64 copy of y before the final rounding
 *   residual_out   : h in the I/O type; required iff residual is given
 *   weight_bias    : added to every weight element (0: the weight itself);
 *                    must be 0 without a weight
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_rmsnorm_rows(const void *x, const void *residual, const void *w,
                        void *y, double *y_exact, void *residual_out,
                        int64_t row_begin, int64_t row_end, int64_t hidden,
                        float eps, float weight_bias, int dtype)
{
    if (x == NULL || y == NULL || hidden <= 0 || row_begin < 0 || row_end < row_begin)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16)
        return -1;
    if ((residual == NULL) != (residual_out == NULL))
        return -1;
    if (w == NULL && weight_bias != 0.0f)
        return -1;
    double *v = (double *)malloc((size_t)hidden * sizeof(double));
    if (v == NULL)
        return -1;
    for (int64_t row = row_begin; row < row_end; ++row) {
        rms_row_values(x, residual, w, row, hidden, (double)eps, (double)weight_bias, dtype, v,
                       residual_out);
        for (int64_t i = 0; i < hidden; ++i) {
            if (y_exact != NULL)
                y_exact[row * hidden + i] = v[i];
            store_elem(y, row * hidden + i, dtype, v[i]);   /* one rounding to the I/O type */
        }
    }
    free(v);
    return 0;
}

/*
 * RMSNorm in the eager framework's op-by-op cast order, rows [row_begin,
 * row_end).  "model-as-a-kernel" (sections "Method" and "Correctness") keeps
 * the eager framework's bf16 semantics op for op and matches its fused
 * rmsnorm bitwise; the pages give no cast order for the norm, and the reading
 * taken is the one of a norm whose weight multiply is an op of its own: the
 * normalised value is computed wide, rounded to the I/O type, then multiplied
 * by the weight and rounded again.
 *   v_i   = h_i * r                          (fp64, as oracle_rmsnorm_rows without w)
 *   n_i   = RN_T(v_i)
 *   y_i   = RN_T(n_i * w_i)                  (n_i without a weight)
 * n_exact (optional) receives v.  Returns 0, or -1 on an invalid argument.
 */
int oracle_rmsnorm_cast_rows(const void *x, const void *residual, const void *w,
                             void *y, double *n_exact, void *residual_out,
                             int64_t row_begin, int64_t row_end, int64_t hidden,
                             float eps, int dtype)
{
    if (x == NULL || y == NULL || hidden <= 0 || row_begin < 0 || row_end < row_begin)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16)
        return -1;
    if ((residual == NULL) != (residual_out == NULL))
        return -1;
    double *v = (double *)malloc((size_t)hidden * sizeof(double));
    if (v == NULL)
        return -1;
    for (int64_t row = row_begin; row < row_end; ++row) {
        rms_row_values(x, residual, NULL, row, hidden, (double)eps, 0.0, dtype, v, residual_out);
        for (int64_t i = 0; i < hidden; ++i) {
            if (n_exact != NULL)
                n_exact[row * hidden + i] = v[i];
            double n = round_to_type(v[i], dtype);            /* the cast to the I/O type */
            if (w != NULL)
                n = n * load_elem(w, i, dtype);              /* exact in binary64 for bf16 and fp32 */
            store_elem(y, row * hidden + i, dtype, n);       /* the weight op's rounding */
        }
    }
    free(v);
    return 0;
}

/*
 * LayerNorm, rows [row_begin, row_end) ("GPT-2 on the GPU", section "The
 * Whole Model as One Kernel": the traced block takes the mean and the
 * variance of the row, normalises as (x - mean) / sqrt(variance + eps) and
 * returns weight * normalised + bias):
 *   h      = x, or RN_T(x + residual) as above
 *   mean   = sum_i h_i / hidden
 *   var    = sum_i (h_i - mean)^2 / hidden        (population variance)
 *   n_i    = (h_i - mean) / sqrt(var + eps)
 *   y_i    = RN_T(w_i * n_i + b_i)                (w, b optional; b needs w)
 * n_exact, y_exact: optional fp64 copies of n and of y before rounding.
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_layernorm_rows(const void *x, const void *residual, const void *w, const void *b,
                          void *y, double *n_exact, double *y_exact, void *residual_out,
                          int64_t row_begin, int64_t row_end, int64_t hidden, float eps, int dtype)
{
    if (x == NULL || y == NULL || hidden <= 0 || row_begin < 0 || row_end < row_begin)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16)
        return -1;
    if ((residual == NULL) != (residual_out == NULL))
        return -1;
    if (b != NULL && w == NULL)
        return -1;

    const double e = (double)eps;
    for (int64_t row = row_begin; row < row_end; ++row) {
        const int64_t base = row * hidden;
        double sum = 0.0;
        for (int64_t i = 0; i < hidden; ++i)
            sum += row_input(x, residual, base + i, dtype);
        const double mean = sum / (double)hidden;
        double sq = 0.0;
        for (int64_t i = 0; i < hidden; ++i) {
            double d = row_input(x, residual, base + i, dtype) - mean;
            sq += d * d;
        }
        const double var = sq / (double)hidden;
        const double denom = sqrt(var + e);
        for (int64_t i = 0; i < hidden; ++i) {
            double h = row_input(x, residual, base + i, dtype);
            double n = (h - mean) / denom;
            double v = n;
            if (w != NULL)
                v = load_elem(w, i, dtype) * n;
            if (b != NULL)
                v = v + load_elem(b, i, dtype);
            if (n_exact != NULL)
                n_exact[base + i] = n;
            if (y_exact != NULL)
                y_exact[base + i] = v;
            store_elem(y, base + i, dtype, v);
            if (residual_out != NULL)
                store_elem(residual_out, base + i, dtype, h);
        }
    }
    return 0;
}

/*
 * FP8 E4M3 (OCP 8-bit floating point): 1 sign bit, 4 exponent bits (bias 7),
 * 3 fraction bits; no infinities; S.1111.111 is NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448; subnormals have the fixed quantum 2^-9.
 * Rounding to E4M3 here: round to nearest, ties to even, on 4 significant
 * bits, then saturate magnitudes above 448 to 448 ("satfinite").
 */
static uint8_t double_to_e4m3_sat(double v)
{
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    if (isnan(v))
        return (uint8_t)(sign | 0x7Fu);
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint8_t)(sign | 0x7Eu);
    int e;
    frexp(a, &e);                 /* a in [2^(e-1), 2^e)                     */
    int q = e - 4;                /* 4 significant bits: quantum 2^(e-1-3)   */
    if (q < -9)
        q = -9;                   /* subnormal quantum                        */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r > 448.0)
        r = 448.0;
    /* encode r (exactly representable) */
    if (r < ldexp(1.0, -6)) {                   /* subnormal: r = m * 2^-9   */
        int m = (int)ldexp(r, 9);
        return (uint8_t)(sign | (uint8_t)m);
    }
    int re;
    double f = frexp(r, &re);                   /* r = f * 2^re, f in [0.5,1) */
    int exp_field = re - 1 + 7;
    int mant = (int)ldexp(f * 2.0 - 1.0, 3);    /* 3 fraction bits            */
    return (uint8_t)(sign | (uint8_t)(exp_field << 3) | (uint8_t)mant);
}

static double e4m3_to_double(uint8_t c)
{
    double s = (c & 0x80u) ? -1.0 : 1.0;
    int ef = (c >> 3) & 0xF;
    int m = c & 0x7;
    if (ef == 0xF && m == 0x7)
        return NAN;
    if (ef == 0)
        return s * ldexp((double)m, -9);
    return s * ldexp(1.0 + m / 8.0, ef - 7);
}

/*
 * RMSNorm with MXFP8 output (OCP Microscaling Formats v1.0, MXFP8 with E4M3
 * elements; block-scaled low-precision output is named in "CuTeDSL at
 * Perplexity", section "Blackwell support").  The op's values v_i (y_i of
 * oracle_rmsnorm_rows before its rounding, weight bias included) are grouped
 * in blocks of 32 consecutive elements of a row.  For each block:
 *   amax   = max_i |v_i|
 *   s      = floor(log2(amax)) - 8, clamped to [-127, 127] (s = -127 when amax is 0)
 *   scale  = E8M0 code s + 127
 *   code_i = E4M3 of v_i / 2^s, nearest-even, saturated at 448
 * A block holding a NaN or an infinity is a NaN block: scale 0xFF (the E8M0
 * NaN) and every code 0x7F (the E4M3 NaN).
 * hidden must be a multiple of 32.  codes [rows, hidden], scales [rows, hidden/32];
 * v_exact (optional) receives the fp64 values.
 */
int oracle_rmsnorm_mxfp8_rows(const void *x, const void *residual, const void *w,
                              uint8_t *codes, uint8_t *scales, double *v_exact, void *residual_out,
                              int64_t row_begin, int64_t row_end, int64_t hidden,
                              float eps, float weight_bias, int dtype)
{
    if (x == NULL || codes == NULL || scales == NULL || hidden <= 0 || hidden % 32 != 0)
        return -1;
    if (row_begin < 0 || row_end < row_begin || (dtype != ORACLE_F32 && dtype != ORACLE_BF16))
        return -1;
    if ((residual == NULL) != (residual_out == NULL) || (w == NULL && weight_bias != 0.0f))
        return -1;
    double *v = (double *)malloc((size_t)hidden * sizeof(double));
    if (v == NULL)
        return -1;
    for (int64_t row = row_begin; row < row_end; ++row) {
        rms_row_values(x, residual, w, row, hidden, (double)eps, (double)weight_bias, dtype, v,
                       residual_out);
        if (v_exact != NULL)
            memcpy(v_exact + row * hidden, v, (size_t)hidden * sizeof(double));
        for (int64_t k = 0; k < hidden / 32; ++k) {
            const double *vb = v + k * 32;
            double amax = 0.0;
            int special = 0;
            for (int j = 0; j < 32; ++j) {
                if (isnan(vb[j]) || isinf(vb[j]))
                    special = 1;
                else if (fabs(vb[j]) > amax)
                    amax = fabs(vb[j]);
            }
            int s = -127;
            if (amax > 0.0) {
                int e;
                frexp(amax, &e);          /* amax in [2^(e-1), 2^e): floor(log2(amax)) = e - 1 */
                s = (e - 1) - 8;          /* 8: exponent of the largest E4M3 value, 1.75 * 2^8  */
                if (s < -127)
                    s = -127;
                if (s > 127)
                    s = 127;
            }
            scales[row * (hidden / 32) + k] = special ? 0xFFu : (uint8_t)(s + 127);
            for (int j = 0; j < 32; ++j)
                codes[row * hidden + k * 32 + j] = special ? 0x7Fu : double_to_e4m3_sat(ldexp(vb[j], -s));
        }
    }
    free(v);
    return 0;
}

/*
 * FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 fraction bit; magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6; no infinities or NaN.  Rounding to E2M1 here:
 * round to nearest on the format's grid (quantum 0.5 below 2, 1 in [2, 4),
 * 2 in [4, 8)), ties to the even code, then saturate above 6 to 6.  The
 * 4-bit code is sign << 3 | magnitude index (0 .. 7 in value order).
 */
static uint8_t double_to_e2m1_sat(double v)
{
    uint8_t sign = signbit(v) ? 0x8u : 0u;
    double a = fabs(v);
    if (isnan(a))
        return 0x7u;                     /* NaN is not encodable: largest positive */
    double q = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double r = nearbyint(a / q) * q;     /* a / q is exact (q a power of two)     */
    if (r > 6.0)
        r = 6.0;
    static const double mags[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint8_t idx = 0;
    for (uint8_t i = 0; i < 8; ++i)
        if (mags[i] == r)
            idx = i;
    return (uint8_t)(sign | idx);
}

static double e2m1_to_double(uint8_t c)
{
    static const double mags[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    return ((c & 0x8u) ? -1.0 : 1.0) * mags[c & 0x7u];
}

/*
 * RMSNorm with NVFP4 output (E2M1 elements, one E4M3 scale per 16 elements,
 * and a per-tensor fp32 scale S given by the caller; the format is named in
 * "CuTeDSL at Perplexity", section "Blackwell support", without a recipe).
 * Reading taken: the value decodes as code * scale * S.  For each block of 16
 * consecutive elements of a row, with the op's values v_i (as for MXFP8):
 *   scale  = E4M3(amax / (6 * S)), nearest-even, saturated at 448
 *   code_i = E2M1(v_i / (scale * S)), nearest-even, saturated at 6
 *            (all codes 0 when the scale is 0)
 * A block holding NaN or Inf gets the E4M3 NaN (0x7F) as its scale and codes 0.
 * codes: [rows, hidden / 2] bytes, element 2k in the low nibble of byte k;
 * scales: [rows, hidden / 16].  hidden must be a multiple of 16; S > 0 finite.
 */
int oracle_rmsnorm_nvfp4_rows(const void *x, const void *residual, const void *w,
                              uint8_t *codes, uint8_t *scales, double *v_exact, void *residual_out,
                              int64_t row_begin, int64_t row_end, int64_t hidden,
                              float eps, float weight_bias, float tensor_scale, int dtype)
{
    if (x == NULL || codes == NULL || scales == NULL || hidden <= 0 || hidden % 16 != 0)
        return -1;
    if (row_begin < 0 || row_end < row_begin || (dtype != ORACLE_F32 && dtype != ORACLE_BF16))
        return -1;
    if ((residual == NULL) != (residual_out == NULL) || (w == NULL && weight_bias != 0.0f))
        return -1;
    if (!(tensor_scale > 0.0f) || isinf(tensor_scale))
        return -1;
    const double S = (double)tensor_scale;
    double *v = (double *)malloc((size_t)hidden * sizeof(double));
    if (v == NULL)
        return -1;
    for (int64_t row = row_begin; row < row_end; ++row) {
        rms_row_values(x, residual, w, row, hidden, (double)eps, (double)weight_bias, dtype, v,
                       residual_out);
        if (v_exact != NULL)
            memcpy(v_exact + row * hidden, v, (size_t)hidden * sizeof(double));
        for (int64_t k = 0; k < hidden / 16; ++k) {
            const double *vb = v + k * 16;
            double amax = 0.0;
            int special = 0;
            for (int j = 0; j < 16; ++j) {
                if (isnan(vb[j]) || isinf(vb[j]))
                    special = 1;
                else if (fabs(vb[j]) > amax)
                    amax = fabs(vb[j]);
            }
            uint8_t sc = special ? 0x7Fu : double_to_e4m3_sat(amax / (6.0 * S));
            scales[row * (hidden / 16) + k] = sc;
            const double sv = special ? 0.0 : e4m3_to_double(sc);
            for (int j = 0; j < 16; j += 2) {
                uint8_t lo = 0, hi = 0;
                if (sv > 0.0) {
                    lo = double_to_e2m1_sat(vb[j] / (sv * S));
                    hi = double_to_e2m1_sat(vb[j + 1] / (sv * S));
                }
                codes[row * (hidden / 2) + (k * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    free(v);
    return 0;
}

void oracle_e2m1_from_double(const double *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = double_to_e2m1_sat(v[i]);
}

void oracle_double_from_e2m1(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = e2m1_to_double(c[i]);
}

void oracle_e4m3_from_double(const double *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = double_to_e4m3_sat(v[i]);
}

void oracle_double_from_e4m3(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_to_double(c[i]);
}

/* Elementwise conversions, exposed so that tests can pin them on their own. */
void oracle_bf16_from_double(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = double_to_bf16(v[i]);
}

void oracle_double_from_bf16(const uint16_t *bits, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_to_double(bits[i]);
}
