/*
 * w8a8_fp8_oracle.c -- plain CPU oracle for the W8A8-FP8 comparison GEMM.
 *
 * TEST INFRASTRUCTURE ONLY (same rules as w4a16_oracle.c: loaded by the
 * tests, the smoke check and the benchmark's CPU legs, never by the product
 * path, and sharing no code with it).
 *
 * What it computes: "Give Me BF16 or Give Me Death" (summary page), section
 * "W8A8-FP Quantization: 8-Bit Floating-Point Weights and Activations":
 *  - paragraph "Weight quantization for FP8": symmetric, one scale per output
 *    channel, s = max|w| / q_max, codes = rnd(w / s), rnd = nearest FP8 value;
 *  - paragraph "Activation quantization for FP8": the same per token (row of
 *    the activation matrix), computed on the fly;
 *  - the quantised weights and activations are multiplied in FP8 on the
 *    tensor cores; the output is y = (s_x q_x) . (s_w q_w).
 *
 * Readings taken where the section is silent (listed in the design notes):
 *  - the FP8 format is E4M3 with no infinities (bias 7, largest finite 448,
 *    smallest subnormal 2^-9), so q_max = 448;
 *  - the scale is a binary32 number, s = fl32(max / 448); the quotient w / s
 *    is a binary32 division and is rounded once to E4M3, ties to even,
 *    saturating at +-448 (a quantised code is a decision both sides take in
 *    the same precision);
 *  - an all-zero row or channel has s = 0 and codes 0;
 *  - orientation: x bf16 [B][K] -> codes [B][K] + scales [B]; W bf16 [K][N]
 *    -> codes [N][K] (one row per output channel) + scales [N];
 *  - GEMM reference value: acc = sum_k dec(q_x) dec(q_w), exact in binary64
 *    (every product of two E4M3 values has at most 8 significant bits and is
 *    a multiple of 2^-18, below 2^17.7 in magnitude, so for K <= 2^15 the sum
 *    needs at most 51 bits); y = RNE_bf16(acc * s_x * s_w);
 *  - error bound: |y_gpu - y| <= 8e-3 * sum_k |s_x dec(q_x) s_w dec(q_w)| + 1e-6,
 *    the same form as the W4A16 bound.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

uint16_t oracle_bf16_from_double(double v);  /* w4a16_oracle.c */

#define FP8_QMAX 448.0

/* E4M3 code -> value: sign, 4-bit exponent field (bias 7), 3-bit fraction;
 * field 0 is subnormal (fraction * 2^-9); 0x7F / 0xFF are NaN. */
double oracle_e4m3_to_double(uint8_t c)
{
    int sign = c >> 7, field = (c >> 3) & 15, frac = c & 7;
    double v;
    if (field == 15 && frac == 7)
        return NAN;
    if (field == 0)
        v = ldexp((double)frac, -9);
    else
        v = ldexp(1.0 + frac / 8.0, field - 7);
    return sign ? -v : v;
}

/* value -> E4M3, round to nearest, ties to an even fraction, saturating to
 * +-448 (no infinities in the format).  Same construction as the bf16
 * encoder: scale to the binade's quantum, rint, rebuild the fields. */
uint8_t oracle_e4m3_from_double(double v)
{
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (a >= FP8_QMAX)
        return (uint8_t)(sign | 0x7E);
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;                       /* a in [2^E, 2^(E+1)) */
    int qexp = (E < -6) ? -9 : E - 3;     /* 3 fraction bits; subnormal quantum 2^-9 */
    double r = rint(ldexp(a, -qexp));
    if (E < -6)
        return (uint8_t)(sign | (uint8_t)r);   /* r == 8 encodes the smallest normal */
    int field = E + 7;
    if (r >= 16.0) {
        r = 8.0;
        field += 1;
    }
    int frac = (int)r - 8;
    if (field > 15 || (field == 15 && frac == 7))
        return (uint8_t)(sign | 0x7E);        /* rounded past 448: saturate */
    return (uint8_t)(sign | (field << 3) | frac);
}

static float bf16_bits_to_float(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Quantise one vector of n bf16 values, element i at v[i * stride]: returns
 * the binary32 scale, writes codes[i]. */
static float quantize_vector(const uint16_t *v, long stride, int n, uint8_t *codes)
{
    float m = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(bf16_bits_to_float(v[(long)i * stride]));
        if (a > m) m = a;
    }
    float s = m / 448.0f;     /* binary32 division (no contraction, no excess precision) */
    for (int i = 0; i < n; ++i) {
        if (s == 0.0f) {
            codes[i] = 0;
            continue;
        }
        float q = bf16_bits_to_float(v[(long)i * stride]) / s;
        codes[i] = oracle_e4m3_from_double((double)q);
    }
    return s;
}

/* Activations, dynamic per token: x bf16 [B][K] -> codes [B][K], scales [B]. */
void oracle_fp8_quantize_rows(const uint16_t *x, int B, int K, uint8_t *codes, float *scales)
{
    for (int b = 0; b < B; ++b)
        scales[b] = quantize_vector(x + (size_t)b * K, 1, K, codes + (size_t)b * K);
}

/* Weights, per output channel: W bf16 [K][N] -> codes [N][K], scales [N]. */
void oracle_fp8_quantize_cols(const uint16_t *w, int K, int N, uint8_t *codes, float *scales)
{
    for (int n = 0; n < N; ++n)
        scales[n] = quantize_vector(w + n, N, K, codes + (size_t)n * K);
}

/* GEMM on a chosen set of output columns:
 *   xq [B][K], sx [B]; wq [N][K], sw [N]; y bf16 bits, acc (exact code sum,
 *   before the scales) and bound, each [B][ncols] (any may be NULL). */
void oracle_fp8_gemm_cols(const uint8_t *xq, const float *sx, const uint8_t *wq,
                          const float *sw, int B, int K, int N, const int *cols, int ncols,
                          uint16_t *y, double *acc, double *bound)
{
    (void)N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int c = 0; c < ncols; ++c) {
        const uint8_t *wr = wq + (size_t)cols[c] * K;
        double s_w = (double)sw[cols[c]];
        for (int b = 0; b < B; ++b) {
            const uint8_t *xr = xq + (size_t)b * K;
            double sum = 0.0, mag = 0.0;
            for (int k = 0; k < K; ++k) {
                double p = oracle_e4m3_to_double(xr[k]) * oracle_e4m3_to_double(wr[k]);
                sum += p;
                mag += fabs(p);
            }
            double s = (double)sx[b] * s_w;
            size_t o = (size_t)b * ncols + c;
            if (y)
                y[o] = oracle_bf16_from_double(sum * s);
            if (acc)
                acc[o] = sum;
            if (bound)
                bound[o] = 8e-3 * mag * s + 1e-6;
        }
    }
}
