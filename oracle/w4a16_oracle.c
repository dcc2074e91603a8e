/*
 * w4a16_oracle.c -- plain CPU oracle for the W4A16 group-128 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA library is checked against.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never does, and this file shares no code, header or table with it.
 *
 * What it computes (sources, by page title and section):
 *  - "Give Me BF16 or Give Me Death" (summary page), section "W4A16-INT
 *    Quantization", paragraph "Group-wise quantization granularity": every 128
 *    consecutive weights along the input dimension K share one 16-bit scale.
 *  - same section, paragraph "Inference with W4A16": the weight is rebuilt as
 *    scale times integer code and the product with the 16-bit activations is
 *    accumulated in higher precision.
 *  - "When quantization pays -- and when it does not", section "Counting c from
 *    the kernel, not from intuition": the code is unsigned 4-bit with bias 8
 *    (the subtracted constant is bf16 136 = 128 + 8), the integer (q - 8) is
 *    formed exactly first and the bf16 group scale is applied after it with
 *    one bf16 multiply.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *  - orientation y[B][N] = x[B][K] . W[K][N], groups run along K;
 *  - bf16 activations, scales and output;
 *  - dequantised weight w = RNE_bf16((q - z) * s), one rounding of the exact
 *    product, z = 8 for the symmetric format, z a stored 4-bit zero-point for
 *    the asymmetric variant;
 *  - canonical code layout: qweight is uint32 [K/8][N], nibble j (bits 4j..4j+3)
 *    of word [kk][n] is the code of row k = 8*kk + j, column n;
 *  - zero-point layout: qzeros is uint32 [K/128][N/8], nibble j of word [g][nn]
 *    is the zero-point of group g, column 8*nn + j;
 *  - GEMM reference value: acc = sum over k, in k order, of double(x) * double(w);
 *    y = RNE_bf16(acc);
 *  - error bound: |y_gpu - y| <= 8e-3 * sum_k |x * w| + 1e-6.
 *
 * Every floating-point step here is written out from its definition: bf16 is
 * the upper half of an IEEE-754 binary32, and RNE_bf16 rounds an exact double
 * to the nearest bf16 with ties to an even significand, overflowing to
 * infinity, with gradual underflow.  No step uses binary32 arithmetic, so no
 * value is rounded twice.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_GROUP 128

#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads for the OpenMP loops below (the CPU-baseline timing runs the oracle
 * on all host cores and on one). */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}

/* bf16 -> double: the 16 bits are the top half of a binary32, which a double
 * holds exactly. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* double -> bf16, round to nearest, ties to even, in one rounding step.
 * bf16 has 8 significand bits (7 stored), exponent bias 127, smallest normal
 * 2^-126, subnormal spacing 2^-133, largest finite (2 - 2^-7) * 2^127. */
uint16_t oracle_bf16_from_double(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);

    int e2;
    (void)frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;               /* a in [2^E, 2^(E+1)) */
    /* quantum = spacing of bf16 numbers at a's binade; below 2^-126 the
     * spacing stays at the subnormal quantum 2^-133. */
    int qexp = (E < -126) ? -133 : E - 7;
    double r = rint(ldexp(a, -qexp));   /* exact scaling; rint = ties-to-even */

    if (E < -126) {
        /* subnormal: r in [0, 128]; r == 128 is the smallest normal, whose
         * encoding (exponent field 1, fraction 0) is again just r. */
        return (uint16_t)(sign | (uint16_t)r);
    }
    /* normal: r in [128, 256]; 256 carries into the next binade. */
    int expo = E;
    if (r >= 256.0) {
        r = 128.0;
        expo = E + 1;
    }
    if (expo > 127)
        return (uint16_t)(sign | 0x7F80u);            /* overflow -> inf */
    uint16_t field = (uint16_t)(expo + 127);
    uint16_t frac = (uint16_t)((int)r - 128);
    return (uint16_t)(sign | (uint16_t)(field << 7) | frac);
}

/* Element-wise oracle_bf16_from_double over an array. */
void oracle_bf16_from_double_array(const double *v, long long n, uint16_t *out)
{
    for (long long i = 0; i < n; ++i)
        out[i] = oracle_bf16_from_double(v[i]);
}

/* Code of weight (k, n) from the canonical uint32 [K/8][N] array. */
int oracle_code(const uint32_t *qweight, int N, int k, int n)
{
    uint32_t word = qweight[(size_t)(k / 8) * (size_t)N + (size_t)n];
    return (int)((word >> (4 * (k % 8))) & 0xFu);
}

/* Zero-point of (group g, column n) from uint32 [K/128][N/8], or the bias 8 of
 * the symmetric format when qzeros is NULL. */
int oracle_zero(const uint32_t *qzeros, int N, int g, int n)
{
    if (qzeros == NULL)
        return 8;
    uint32_t word = qzeros[(size_t)g * (size_t)(N / 8) + (size_t)(n / 8)];
    return (int)((word >> (4 * (n % 8))) & 0xFu);
}

/* One dequantised weight: RNE_bf16((q - z) * s).  The product of an integer of
 * magnitude <= 15 and a bf16 value is exact in double, so this is the single
 * rounding of the exact value. */
uint16_t oracle_dequant_one(int q, int z, uint16_t scale_bits)
{
    double s = oracle_bf16_to_double(scale_bits);
    return oracle_bf16_from_double((double)(q - z) * s);
}

/* Materialise W[K][N] as bf16 bits. */
void oracle_dequant(const uint32_t *qweight, const uint16_t *scales,
                    const uint32_t *qzeros, int K, int N, uint16_t *w_out)
{
#pragma omp parallel for schedule(static)
    for (int k = 0; k < K; ++k) {
        int g = k / ORACLE_GROUP;
        for (int n = 0; n < N; ++n) {
            int q = oracle_code(qweight, N, k, n);
            int z = oracle_zero(qzeros, N, g, n);
            w_out[(size_t)k * N + n] =
                oracle_dequant_one(q, z, scales[(size_t)g * N + n]);
        }
    }
}

/* GEMM on a chosen set of output columns.
 *   x       bf16 bits [B][K]
 *   cols    ncols column indices into N (all of them for a full check)
 *   y       bf16 bits [B][ncols]          (may be NULL)
 *   acc     double    [B][ncols]          unrounded sum      (may be NULL)
 *   bound   double    [B][ncols]          8e-3*sum|x*w|+1e-6 (may be NULL)
 * For each requested column the K dequantised weights are formed first, then
 * every batch row is a plain dot product summed in k order. */
void oracle_gemm_cols(const uint16_t *x, const uint32_t *qweight,
                      const uint16_t *scales, const uint32_t *qzeros,
                      int B, int K, int N, const int *cols, int ncols,
                      uint16_t *y, double *acc, double *bound)
{
#pragma omp parallel
    {
        double *wcol = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
        for (int c = 0; c < ncols; ++c) {
            int n = cols[c];
            for (int k = 0; k < K; ++k) {
                int g = k / ORACLE_GROUP;
                uint16_t wb = oracle_dequant_one(oracle_code(qweight, N, k, n),
                                                 oracle_zero(qzeros, N, g, n),
                                                 scales[(size_t)g * N + n]);
                wcol[k] = oracle_bf16_to_double(wb);
            }
            for (int b = 0; b < B; ++b) {
                const uint16_t *xr = x + (size_t)b * K;
                double sum = 0.0, mag = 0.0;
                for (int k = 0; k < K; ++k) {
                    double p = oracle_bf16_to_double(xr[k]) * wcol[k];
                    sum += p;
                    mag += fabs(p);
                }
                size_t o = (size_t)b * ncols + c;
                if (y)
                    y[o] = oracle_bf16_from_double(sum);
                if (acc)
                    acc[o] = sum;
                if (bound)
                    bound[o] = 8e-3 * mag + 1e-6;
            }
        }
        free(wcol);
    }
}

/* Size of the stored format in bytes (codes + scales [+ zero-points]), the
 * quantity behind the 4.125 effective bits per weight of the group-128
 * format. */
double oracle_format_bits_per_weight(long long K, long long N, int has_zeros)
{
    long long groups = K / ORACLE_GROUP;
    double code_bytes = (double)(K * N) / 2.0;      /* 4 bits per code */
    double scale_bytes = (double)(groups * N) * 2.0; /* one bf16 per group */
    double zero_bytes = has_zeros ? (double)(groups * N) / 2.0 : 0.0;
    return (code_bytes + scale_bytes + zero_bytes) * 8.0 / (double)(K * N);
}

/* ------------------------------------------------------------------------
 * Offline quantizer: round to nearest with MSE-optimal clipping.
 *
 * "Give Me BF16 or Give Me Death" (summary page), section "W4A16-INT
 * Quantization", paragraph "Weight quantization algorithm: GPTQ with
 * MSE-optimal clipping": for each group of 128 consecutive weights (along K,
 * per output column), search a clipping ratio alpha on a grid; the scale is
 * alpha * max|x| / 7, a weight is rounded to the nearest multiple of the scale
 * and saturated to [-7, 7] (symmetric signed INT4, -8 unused), and the alpha
 * with the smallest sum of squared errors sum (x - Q_alpha(x))^2 is kept.  The
 * GPTQ Hessian update needs calibration data and is not part of this path.
 *
 * Readings (the pages leave these open; listed in the design notes):
 *  - grid alpha_i = 1 - i/32, i = 0 .. 23 (1 down to 0.28125), every
 *    alpha * max exact in binary32;
 *  - the scale is stored as bf16, so it is rounded (RNE) before the codes are
 *    chosen, and the error is measured on the weights the GEMM will see,
 *    RNE_bf16(code * scale);
 *  - code = clamp(round_half_even(x / s), -7, 7), stored with bias 8;
 *  - the divisions and the rounding to an integer are binary32 operations, as
 *    in the kernel (a quantised code is a decision both sides must take in the
 *    same precision); x - Q(x) is exact in binary32 (both are bf16 values at
 *    most a few binades apart, or Q(x) = 0) and its square exact in binary64;
 *    the error is summed in binary64 in k order;
 *  - ties between grid points keep the earlier (larger) alpha; a group of
 *    zeros gets scale 0 and codes 8.
 * Inputs: w bf16 [K][N] (row k, column n).  Outputs: canonical qweight uint32
 * [K/8][N] and scales bf16 [K/128][N].
 */
#define ORACLE_QGRID 24

static float oracle_bf16_to_float(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

void oracle_quantize_rtn_mse(const uint16_t *w, int K, int N, uint32_t *qweight,
                             uint16_t *scales)
{
    memset(qweight, 0, (size_t)(K / 8) * (size_t)N * sizeof(uint32_t));
    for (int g = 0; g < K / ORACLE_GROUP; ++g) {
        for (int n = 0; n < N; ++n) {
            float m = 0.0f;
            for (int r = 0; r < ORACLE_GROUP; ++r) {
                float v = fabsf(oracle_bf16_to_float(w[(size_t)(g * ORACLE_GROUP + r) * N + n]));
                if (v > m) m = v;
            }
            int best = -1;
            double best_err = 0.0;
            uint16_t best_s = 0;
            for (int i = 0; i < ORACLE_QGRID; ++i) {
                float alpha = 1.0f - (float)i / 32.0f;
                float sf = (alpha * m) / 7.0f;
                uint16_t sb = oracle_bf16_from_double((double)sf);
                float s = oracle_bf16_to_float(sb);
                if (!(s > 0.0f)) continue;
                double err = 0.0;
                for (int r = 0; r < ORACLE_GROUP; ++r) {
                    float x = oracle_bf16_to_float(w[(size_t)(g * ORACLE_GROUP + r) * N + n]);
                    float q = rintf(x / s);
                    if (q > 7.0f) q = 7.0f;
                    if (q < -7.0f) q = -7.0f;
                    float xq = oracle_bf16_to_float(oracle_dequant_one((int)q + 8, 8, sb));
                    float e = x - xq;
                    err += (double)e * (double)e;
                }
                if (best < 0 || err < best_err) {
                    best = i;
                    best_err = err;
                    best_s = sb;
                }
            }
            scales[(size_t)g * N + n] = best < 0 ? 0 : best_s;
            for (int r = 0; r < ORACLE_GROUP; ++r) {
                int code = 8;
                if (best >= 0) {
                    float x = oracle_bf16_to_float(w[(size_t)(g * ORACLE_GROUP + r) * N + n]);
                    float q = rintf(x / oracle_bf16_to_float(best_s));
                    if (q > 7.0f) q = 7.0f;
                    if (q < -7.0f) q = -7.0f;
                    code = (int)q + 8;
                }
                int k = g * ORACLE_GROUP + r;
                qweight[(size_t)(k / 8) * N + n] |= (uint32_t)code << (4 * (k % 8));
            }
        }
    }
}
