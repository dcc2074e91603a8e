/*
 * w4a16_f16_oracle.c -- plain CPU oracle for the fp16-activation variant of
 * the W4A16 group-128 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY, like w4a16_oracle.c beside it: the slow, plainly
 * written definition the CUDA library's fp16 entry points are checked
 * against.  It shares no code, header or table with the library.
 *
 * What it computes (sources, by page title and section):
 *  - "Give Me BF16 or Give Me Death" (summary page), section "W4A16-INT
 *    Quantization", paragraph "Inference with W4A16": the dequantised weights,
 *    the scales and the tensor-core products are 16-bit floating point -- the
 *    paragraph names fp16 -- with the products accumulated in higher
 *    precision.  This file is that reading with IEEE-754 binary16 for the
 *    activations, the group scales, the dequantised weights and the output.
 *  - the same section, paragraph "Group-wise quantization granularity": one
 *    scale per 128 consecutive weights along K.
 *  - "When quantization pays -- and when it does not", section "Counting c from
 *    the kernel, not from intuition": uint4 codes with bias 8, the integer
 *    (q - z) formed exactly before the one multiply by the group scale.
 *
 * Readings (listed in the design notes of the repository):
 *  - code and zero-point layouts, orientation and grouping exactly as the bf16
 *    oracle's (canonical qweight uint32 [K/8][N], qzeros uint32 [K/128][N/8]);
 *  - dequantised weight w = RNE_f16((q - z) * s), one rounding of the exact
 *    product;
 *  - reference value acc = sum over k, in k order, of double(x) * double(w);
 *    y = RNE_f16(acc);
 *  - error bound |y_gpu - y| <= 2e-3 * sum_k |x * w| + 2^-24 * (1 + sum_k |x|):
 *    two fp16 unit roundoffs (2^-11 each: the output rounding, and the
 *    weight rounding a kernel that scales the fp32 group sum skips) plus room
 *    for fp32 accumulation, and an absolute term of one fp16 subnormal step
 *    per unit of sum |x| for weights and results below the normal range.
 *
 * binary16: sign bit, 5-bit exponent with bias 15, 10 stored fraction bits;
 * exponent field 0 holds zero and the subnormals (fraction * 2^-24), field 31
 * infinity and NaN; largest finite 65504; round to nearest, ties to even,
 * overflowing to infinity.  Every step below is written from that definition;
 * no step uses binary32 arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#define F16_GROUP 128

/* binary16 bits -> double (exact: 11 significand bits fit a double). */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int field = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    double v;
    if (field == 0)
        v = ldexp((double)frac, -24);              /* zero and subnormals */
    else if (field == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), field - 25);  /* (1 + f/1024) * 2^(field-15) */
    return sign ? -v : v;
}

/* double -> binary16, round to nearest with ties to even, in one step.
 * 11 significand bits (10 stored), smallest normal 2^-14, subnormal spacing
 * 2^-24, largest finite (2 - 2^-10) * 2^15 = 65504. */
uint16_t oracle_f16_from_double(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFE00u : 0x7E00u);
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7C00u);

    int e2;
    (void)frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;               /* a in [2^E, 2^(E+1)) */
    /* spacing of binary16 numbers in a's binade; below 2^-14 it stays at
     * the subnormal spacing 2^-24 */
    int qexp = (E < -14) ? -24 : E - 10;
    double r = rint(ldexp(a, -qexp));   /* exact scaling; rint = ties-to-even */

    if (E < -14) {
        /* subnormal: r in [0, 1024]; r == 1024 is the smallest normal, whose
         * encoding (field 1, fraction 0) is again just r */
        return (uint16_t)(sign | (uint16_t)r);
    }
    /* normal: r in [1024, 2048]; 2048 carries into the next binade */
    int expo = E;
    if (r >= 2048.0) {
        r = 1024.0;
        expo = E + 1;
    }
    if (expo > 15)
        return (uint16_t)(sign | 0x7C00u);             /* overflow -> inf */
    uint16_t field = (uint16_t)(expo + 15);
    uint16_t frac = (uint16_t)((int)r - 1024);
    return (uint16_t)(sign | (uint16_t)(field << 10) | frac);
}

/* Element-wise oracle_f16_from_double over an array. */
void oracle_f16_from_double_array(const double *v, long long n, uint16_t *out)
{
    for (long long i = 0; i < n; ++i)
        out[i] = oracle_f16_from_double(v[i]);
}

static int f16_code(const uint32_t *qweight, int N, int k, int n)
{
    uint32_t word = qweight[(size_t)(k / 8) * (size_t)N + (size_t)n];
    return (int)((word >> (4 * (k % 8))) & 0xFu);
}

static int f16_zero(const uint32_t *qzeros, int N, int g, int n)
{
    if (qzeros == NULL)
        return 8;
    uint32_t word = qzeros[(size_t)g * (size_t)(N / 8) + (size_t)(n / 8)];
    return (int)((word >> (4 * (n % 8))) & 0xFu);
}

/* One dequantised weight: RNE_f16((q - z) * s); the product of an integer of
 * magnitude <= 15 and a binary16 value is exact in double. */
uint16_t oracle_dequant_one_f16(int q, int z, uint16_t scale_bits)
{
    return oracle_f16_from_double((double)(q - z) * oracle_f16_to_double(scale_bits));
}

/* Materialise W[K][N] as binary16 bits. */
void oracle_dequant_f16(const uint32_t *qweight, const uint16_t *scales,
                        const uint32_t *qzeros, int K, int N, uint16_t *w_out)
{
#pragma omp parallel for schedule(static)
    for (int k = 0; k < K; ++k) {
        int g = k / F16_GROUP;
        for (int n = 0; n < N; ++n)
            w_out[(size_t)k * N + n] = oracle_dequant_one_f16(
                f16_code(qweight, N, k, n), f16_zero(qzeros, N, g, n),
                scales[(size_t)g * N + n]);
    }
}

/* GEMM on a chosen set of output columns, fp16 throughout.
 *   x       binary16 bits [B][K]
 *   cols    ncols column indices into N
 *   y       binary16 bits [B][ncols]   (may be NULL)
 *   acc     double [B][ncols], the unrounded sum   (may be NULL)
 *   bound   double [B][ncols], 2e-3*sum|x*w| + 2^-24*(1 + sum|x|)   (may be NULL)
 * For each requested column its K weights are dequantised first; every batch
 * row is then a plain dot product summed in k order. */
void oracle_gemm_cols_f16(const uint16_t *x, const uint32_t *qweight,
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
                int g = k / F16_GROUP;
                wcol[k] = oracle_f16_to_double(oracle_dequant_one_f16(
                    f16_code(qweight, N, k, n), f16_zero(qzeros, N, g, n),
                    scales[(size_t)g * N + n]));
            }
            for (int b = 0; b < B; ++b) {
                const uint16_t *xr = x + (size_t)b * K;
                double sum = 0.0, mag = 0.0, xmag = 0.0;
                for (int k = 0; k < K; ++k) {
                    double xv = oracle_f16_to_double(xr[k]);
                    double p = xv * wcol[k];
                    sum += p;
                    mag += fabs(p);
                    xmag += fabs(xv);
                }
                size_t o = (size_t)b * ncols + c;
                if (y)
                    y[o] = oracle_f16_from_double(sum);
                if (acc)
                    acc[o] = sum;
                if (bound)
                    bound[o] = 2e-3 * mag + ldexp(1.0 + xmag, -24);
            }
        }
        free(wcol);
    }
}
