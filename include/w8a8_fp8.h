/* w8a8_fp8.h -- C ABI of the W8A8-FP8 comparison path in libw4a16.so.
 *
 * "Give Me BF16 or Give Me Death" (summary page), section "W8A8-FP
 * Quantization: 8-Bit Floating-Point Weights and Activations": weights are
 * quantised once per output channel and activations per token at run time,
 * both symmetric with s = max|v| / q_max and codes = the nearest FP8 value of
 * v / s; the product runs on FP8 tensor cores.  "When quantization pays -- and
 * when it does not" (the three regimes) compares this format with W4A16 and
 * bf16 across batch sizes; this path exists to measure that comparison on the
 * same GPU.
 *
 * Format and readings: E4M3 (OCP FP8, no infinities, q_max = 448); scales are
 * binary32; a quotient v / s is a binary32 division rounded once to E4M3
 * (nearest, ties to even, saturating at +-448); an all-zero row or channel
 * gets scale 0 and codes 0.
 *
 * All pointers are device pointers owned by the caller; every call only
 * enqueues work on `stream` (a cudaStream_t, NULL = legacy default stream) and
 * returns a w4a16_status (see w4a16.h) after validating on the host:
 * SHAPE (K % 128 != 0, N % 8 != 0, B < 1), NULL, ALIGN (16 bytes for code,
 * bf16 and workspace buffers; 4 bytes for the fp32 scales), UNSUPPORTED (no
 * tcgen05 tensor cores: GEMM only), WORKSPACE, CUDA.  Device-side waits are
 * bounded; an expired wait sets the status word read by w4a16_device_status.
 */
#ifndef W8A8_FP8_H
#define W8A8_FP8_H

#include <stddef.h>

#include "w4a16.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Dynamic per-token activation quantisation:
 *   x  bf16 [B][K] row-major  ->  xq E4M3 codes uint8 [B][K], sx fp32 [B]. */
w4a16_status w8a8_fp8_quantize_act(const void *x, int B, int K, void *xq, float *sx,
                                   void *stream);

/* Per-output-channel weight quantisation (offline):
 *   w  bf16 [K][N] row-major  ->  wq E4M3 codes uint8 [N][K] (one row per output
 *   channel, the K-major layout the GEMM reads), sw fp32 [N]. */
w4a16_status w8a8_fp8_quantize_weight(const void *w, int K, int N, void *wq, float *sw,
                                      void *stream);

/* Bytes of the GEMM's weight layout: ceil(N/128) * 128 * K. */
size_t w8a8_fp8_packed_bytes(int K, int N);

/* Reorder the [N][K] codes into the GEMM's layout: tiles of 128 channels x
 * 128 k, each one contiguous 16 KB block holding the shared-memory image the
 * MMA reads (128-byte rows, 128-byte swizzle), tile t / k block kb at block
 * t * (K/128) + kb, channels past N zero.  A pure byte permutation.
 *   wq      device uint8 [N][K] (from w8a8_fp8_quantize_weight)   (read)
 *   packed  device, w8a8_fp8_packed_bytes(K, N) bytes             (written) */
w4a16_status w8a8_fp8_pack_weight(const void *wq, int K, int N, void *packed, void *stream);

/* Workspace bytes w8a8_fp8_gemm needs for this shape (0: none; SIZE_MAX for an
 * invalid shape).  Same contract as w4a16_gemm's: zero-filled once by the
 * caller, left zero by every call, shareable with the W4A16 calls. */
size_t w8a8_fp8_workspace_bytes(int B, int K, int N);

/* y[b][n] = bf16( sum_k dec(xq[b][k]) * dec(wq[n][k]) * sx[b] * sw[n] ), fp32
 * accumulation on the tensor cores (tcgen05.mma kind::f8f6f4), bf16 y [B][N];
 * the weight codes are read from `packed` (w8a8_fp8_pack_weight). */
w4a16_status w8a8_fp8_gemm(const void *xq, const float *sx, const void *packed, const float *sw,
                           void *y, int B, int K, int N, void *workspace, size_t ws_bytes,
                           void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_FP8_H */
