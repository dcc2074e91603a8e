// fmt16.cuh -- the two 16-bit floating-point formats the GEMMs run in.
//
// bf16 is the default.  fp16 is the form the "Inference with W4A16"
// paragraph of "Give Me BF16 or Give Me Death" ("W4A16-INT Quantization")
// describes: fp16 activations, group scales, dequantised weights and output,
// products accumulated in fp32.  Each format supplies what differs between
// the two:
//   * the magic-number decode ("When quantization pays -- and when it does
//     not", "Counting c from the kernel, not from intuition"): a 4-bit code q
//     OR-ed into the low fraction bits of a power of two P with at least 4
//     fraction bits gives exactly P + q -- P = 128 (bf16 0x4300, 7 fraction
//     bits) or P = 1024 (fp16 0x6400, 10 fraction bits) -- and subtracting
//     P + z gives the exact integer q - z;
//   * the packed 16-bit arithmetic (sub, mul with round-to-nearest-even);
//   * conversion to and from fp32;
//   * the operand-type codes of the tensor-core instructions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace w4a16 {

struct Bf16 {
    static constexpr bool kIsF16 = false;
    static constexpr uint32_t kMagic2 = 0x43004300u;    // 128.0 in both halves
    static constexpr uint32_t kSymZero2 = 0x43084308u;  // 136.0 = 128 + 8
    static constexpr uint32_t kTcFormat = 1u;           // tcgen05 kind::f16 operand code
    __device__ static __forceinline__ uint32_t sub2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ static __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ static __forceinline__ float to_f32(uint32_t h) {
        return __uint_as_float((h & 0xFFFFu) << 16);
    }
    __device__ static __forceinline__ uint32_t from_f32(float v) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        return *reinterpret_cast<const uint16_t*>(&h);
    }
};

struct F16 {
    static constexpr bool kIsF16 = true;
    static constexpr uint32_t kMagic2 = 0x64006400u;    // 1024.0 in both halves
    static constexpr uint32_t kSymZero2 = 0x64086408u;  // 1032.0 = 1024 + 8
    static constexpr uint32_t kTcFormat = 0u;
    __device__ static __forceinline__ uint32_t sub2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ static __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ static __forceinline__ float to_f32(uint32_t h) {
        return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
    }
    __device__ static __forceinline__ uint32_t from_f32(float v) {
        return __half_as_ushort(__float2half_rn(v));
    }
};

}  // namespace w4a16
