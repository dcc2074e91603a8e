// epilogue.cuh -- fused output epilogues of the W4A16 GEMM kernels.
//
// A linear layer's output usually goes straight into a bias add or, for the
// gate and up projections of a gated MLP, into SiLU(gate) * up.  Applying
// them where the fp32 sums are converted to bf16 saves a separate kernel and
// a round trip of y through HBM.
//   bias      y[b][n] = bf16(acc[b][n] + bias[n]),  bias bf16 [N];
//   silu_mul  columns are interleaved (2j = gate j, 2j+1 = up j) and
//             y[b][j] = bf16(silu(g) * u) with g, u the (biased) fp32 sums of
//             columns 2j and 2j+1 and silu(g) = g / (1 + exp(-g));
//             y is [B][N/2].
// With a K split the bias and the activation are applied once, by the unit
// that converts the finished fp32 sum.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "fmt16.cuh"
#include "launch.cuh"

namespace w4a16 {

// (Epilogue, kEpiBias and kEpiSiluMul are declared in launch.cuh.)

__device__ __forceinline__ float epi_bf16_to_f32(uint32_t h) {
    return __uint_as_float((h & 0xFFFFu) << 16);
}

__device__ __forceinline__ uint32_t epi_f32_to_bf16(float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t*>(&h);
}

__device__ __forceinline__ float epi_silu_mul(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// The kernels are compiled with and without the fused forms, so the plain
// kernels carry none of this code.
static __device__ __forceinline__ void epi_store4_fused(uint16_t* y, int N, int b, int n, float v0, float v1,
                                              float v2, float v3, Epilogue e) {
    if (e.mode & kEpiBias) {
        const uint2 bb = *reinterpret_cast<const uint2*>(e.bias + n);
        v0 = __fadd_rn(v0, epi_bf16_to_f32(bb.x));
        v1 = __fadd_rn(v1, epi_bf16_to_f32(bb.x >> 16));
        v2 = __fadd_rn(v2, epi_bf16_to_f32(bb.y));
        v3 = __fadd_rn(v3, epi_bf16_to_f32(bb.y >> 16));
    }
    if (e.mode & kEpiSiluMul) {
        *reinterpret_cast<uint32_t*>(y + (size_t)b * (N / 2) + n / 2) =
            epi_f32_to_bf16(epi_silu_mul(v0, v1)) | (epi_f32_to_bf16(epi_silu_mul(v2, v3)) << 16);
    } else {
        *reinterpret_cast<uint2*>(y + (size_t)b * N + n) =
            make_uint2(epi_f32_to_bf16(v0) | (epi_f32_to_bf16(v1) << 16),
                       epi_f32_to_bf16(v2) | (epi_f32_to_bf16(v3) << 16));
    }
}

// Plain conversion of four consecutive columns n .. n+3 (n % 4 == 0) of row b
// to bf16 or fp16 (fmt16.cuh).
template <class Fmt = Bf16>
__device__ __forceinline__ void epi_store4_plain(uint16_t* y, int N, int b, int n, float v0,
                                                 float v1, float v2, float v3, const Epilogue&) {
    *reinterpret_cast<uint2*>(y + (size_t)b * N + n) =
        make_uint2(Fmt::from_f32(v0) | (Fmt::from_f32(v1) << 16),
                   Fmt::from_f32(v2) | (Fmt::from_f32(v3) << 16));
}

// One column per lane: column n of row b, where n runs over consecutive
// columns across the warp's lanes.  Warp-collective (every lane calls it with
// the same b); `ok` says whether this lane's column exists.  The gate / up
// pair of a SiLU column sits in lanes 2i and 2i + 1.
static __device__ __forceinline__ void epi_store_lane_fused(uint16_t* y, int N, int b, int n,
                                                            float v, bool ok, const Epilogue& e) {
    if ((e.mode & kEpiBias) && ok) v = __fadd_rn(v, epi_bf16_to_f32(e.bias[n]));
    if (e.mode & kEpiSiluMul) {
        const float u = __shfl_xor_sync(0xffffffffu, v, 1);
        if (ok && (n & 1) == 0)
            y[(size_t)b * (N / 2) + n / 2] = (uint16_t)epi_f32_to_bf16(epi_silu_mul(v, u));
    } else if (ok) {
        y[(size_t)b * N + n] = (uint16_t)epi_f32_to_bf16(v);
    }
}


}  // namespace w4a16
