// quantize.cu -- offline INT4 quantizer: round to nearest with MSE-optimal
// clipping, producing the canonical codes and bf16 group scales that
// w4a16_pack consumes.
//
// "Give Me BF16 or Give Me Death" (summary page), section "W4A16-INT
// Quantization", paragraph "Weight quantization algorithm: GPTQ with
// MSE-optimal clipping": per group of 128 consecutive weights along K, search
// the clipping ratio alpha on a grid; scale = alpha * max|x| / 7; a weight is
// rounded to the nearest multiple of the scale and saturated to [-7, 7]
// (symmetric signed INT4, -8 unused); keep the alpha with the smallest sum of
// squared errors.  (GPTQ's Hessian-based update needs calibration data and is
// not part of this path.)
//
// Exactly reproducible decisions:
//  - grid alpha_i = 1 - i/32, i = 0 .. 23; alpha * max is exact in binary32;
//  - the scale is rounded to bf16 (it is stored as bf16) before the codes are
//    chosen, and the error is measured on the weights the GEMM will use,
//    RNE_bf16(code * scale), which is the library's dequantisation;
//  - code = clamp(rint(x / s), -7, 7): IEEE binary32 division and
//    round-half-even, no contraction;
//  - x - Q(x) is exact in binary32, its square exact in binary64, and the
//    squares are summed in binary64 in k order -- so the choice of alpha
//    (ties keep the larger alpha) does not depend on how the work is split.
// One thread per (group, column): the column's 128 weights stay in 64
// registers (bf16 pairs) for the 24 passes; loads and stores are coalesced
// across the threads of a CTA (consecutive columns).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.cuh"

namespace w4a16 {
namespace {

constexpr int kQuantThreads = 128;
constexpr int kQuantGrid = 24;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) {
    return __uint_as_float(h << 16);
}

__device__ __forceinline__ uint32_t float_to_bf16_bits(float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    return (uint32_t)*reinterpret_cast<const uint16_t*>(&b);
}

// clamp(rint(x / s), -7, 7)
__device__ __forceinline__ float quant_step(float x, float s) {
    const float q = rintf(__fdiv_rn(x, s));
    return fminf(fmaxf(q, -7.0f), 7.0f);
}

__global__ void __launch_bounds__(kQuantThreads)
quantize_kernel(const uint16_t* __restrict__ w, int N, uint32_t* __restrict__ qweight,
                uint16_t* __restrict__ scales) {
    const int g = blockIdx.y;
    const int n = blockIdx.x * kQuantThreads + threadIdx.x;
    if (n >= N) return;
    const uint16_t* col = w + (size_t)g * kGroup * N + n;
    uint32_t v[kGroup / 2];  // rows (2j, 2j+1) in the low and high halves
#pragma unroll
    for (int j = 0; j < kGroup / 2; ++j)
        v[j] = (uint32_t)__ldg(col + (size_t)(2 * j) * N) |
               ((uint32_t)__ldg(col + (size_t)(2 * j + 1) * N) << 16);
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < kGroup / 2; ++j)
        m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_float(v[j] & 0xFFFFu)),
                           fabsf(bf16_bits_to_float(v[j] >> 16))));
    int best = -1;
    double best_err = 0.0;
    uint32_t best_s = 0;
    for (int i = 0; i < kQuantGrid; ++i) {
        const float alpha = 1.0f - (float)i / 32.0f;
        const uint32_t sb = float_to_bf16_bits(__fdiv_rn(__fmul_rn(alpha, m), 7.0f));
        const float s = bf16_bits_to_float(sb);
        if (!(s > 0.0f)) continue;
        double err = 0.0;
#pragma unroll
        for (int j = 0; j < kGroup / 2; ++j) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float x = bf16_bits_to_float(h ? v[j] >> 16 : v[j] & 0xFFFFu);
                const float xq =
                    bf16_bits_to_float(float_to_bf16_bits(__fmul_rn(quant_step(x, s), s)));
                const float e = __fsub_rn(x, xq);
                err = __dadd_rn(err, __dmul_rn((double)e, (double)e));
            }
        }
        if (best < 0 || err < best_err) {
            best = i;
            best_err = err;
            best_s = sb;
        }
    }
    scales[(size_t)g * N + n] = (uint16_t)(best < 0 ? 0u : best_s);
    const float s = bf16_bits_to_float(best_s);
#pragma unroll
    for (int word = 0; word < kGroup / 8; ++word) {
        uint32_t packed = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t pair = v[(8 * word + t) >> 1];
            const float x = bf16_bits_to_float(t & 1 ? pair >> 16 : pair & 0xFFFFu);
            const int code = best < 0 ? 8 : (int)quant_step(x, s) + 8;
            packed |= (uint32_t)code << (4 * t);
        }
        qweight[(size_t)(g * (kGroup / 8) + word) * N + n] = packed;
    }
}

}  // namespace

cudaError_t launch_quantize(const void* w, int K, int N, uint32_t* qweight, void* scales,
                            cudaStream_t stream) {
    const dim3 grid((N + kQuantThreads - 1) / kQuantThreads, K / kGroup);
    quantize_kernel<<<grid, kQuantThreads, 0, stream>>>(static_cast<const uint16_t*>(w), N,
                                                        qweight, static_cast<uint16_t*>(scales));
    return cudaGetLastError();
}

}  // namespace w4a16
