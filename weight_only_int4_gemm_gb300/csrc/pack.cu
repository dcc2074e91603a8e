// pack.cu -- offline repack of canonical codes into the packed layout, and
// the reference dequantisation kernel that materialises W[K][N].
#include <cuda_runtime.h>

#include "dequant.cuh"
#include "launch.cuh"

namespace w4a16 {
namespace {

constexpr int kPackThreads = 256;

// One thread per (chunk c, column n): gathers the four canonical words of rows
// 32c .. 32c+31 of column n and moves every code to its packed nibble.
__global__ void __launch_bounds__(kPackThreads)
repack_kernel(const uint32_t* __restrict__ qweight, uint4* __restrict__ packed, int K, int N,
              uint4* __restrict__ tag, uint4 tag_value) {
    const int n = blockIdx.x * kPackThreads + threadIdx.x;
    const int c = blockIdx.y;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *tag = tag_value;
    if (n >= N) return;
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t w = __ldg(qweight + (size_t)(4 * c + j) * N + n);
        uint32_t p = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) p |= ((w >> (4 * r)) & 0xFu) << (4 * packed_nibble_of_row(r));
        out[j] = p;
    }
    packed[packed_index16(K, N, c, n)] = make_uint4(out[0], out[1], out[2], out[3]);
}

// One thread per (chunk c, column n): decodes 32 weights with the shared
// routine and writes them to W[32c .. 32c+31][n] (bf16 or fp16, fmt16.cuh).
template <bool kHasZeros, class Fmt>
__global__ void __launch_bounds__(kPackThreads)
dequant_ref_kernel(const uint4* __restrict__ packed, const uint16_t* __restrict__ scales,
                   const uint32_t* __restrict__ zeros, uint16_t* __restrict__ w, int K, int N) {
    const int n = blockIdx.x * kPackThreads + threadIdx.x;
    const int c = blockIdx.y;
    if (n >= N) return;
    const int g = c >> 2;  // 4 chunks of 32 rows per group of 128
    const uint4 q = packed[packed_index16(K, N, c, n)];
    const uint32_t s2 = scale_pair(__ldg(scales + (size_t)g * N + n));
    const uint32_t z2 = kHasZeros ? zero_pair<Fmt>(load_zero(zeros, N, g, n)) : Fmt::kSymZero2;
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t pairs[4];
        dequant_word<Fmt>(words[j], z2, s2, pairs);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const size_t k = (size_t)32 * c + 8 * j + 2 * i;
            w[k * N + n] = (uint16_t)(pairs[i] & 0xFFFFu);
            w[(k + 1) * N + n] = (uint16_t)(pairs[i] >> 16);
        }
    }
}

}  // namespace

cudaError_t launch_repack(const uint32_t* qweight, const uint32_t* qzeros, int K, int N,
                          void* packed, cudaStream_t stream) {
    dim3 grid((N + kPackThreads - 1) / kPackThreads, K / 32);
    const BlobTag t = blob_tag(K, N, qzeros != nullptr);
    uint4* tag = reinterpret_cast<uint4*>(static_cast<char*>(packed) +
                                          packed_tag_offset(K, N, qzeros != nullptr));
    repack_kernel<<<grid, kPackThreads, 0, stream>>>(qweight, static_cast<uint4*>(packed), K, N,
                                                     tag, make_uint4(t.w[0], t.w[1], t.w[2], t.w[3]));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || qzeros == nullptr) return err;
    // zero-points: one group per row, rows padded with zero words to 16 bytes
    char* zdst = static_cast<char*>(packed) + packed_code_bytes(K, N);
    err = cudaMemsetAsync(zdst, 0, packed_zero_bytes(K, N), stream);
    if (err != cudaSuccess) return err;
    const size_t row_bytes = (size_t)(N / 8) * 4;
    return cudaMemcpy2DAsync(zdst, (size_t)packed_zero_row_words(N) * 4, qzeros, row_bytes,
                             row_bytes, (size_t)(K / 128), cudaMemcpyDeviceToDevice, stream);
}

cudaError_t launch_dequant_ref(const void* packed, const void* scales, bool has_zeros, void* w,
                               int K, int N, bool f16, cudaStream_t stream) {
    dim3 grid((N + kPackThreads - 1) / kPackThreads, K / 32);
    const uint4* p = static_cast<const uint4*>(packed);
    const uint16_t* s = static_cast<const uint16_t*>(scales);
    const uint32_t* z = reinterpret_cast<const uint32_t*>(static_cast<const char*>(packed) +
                                                          packed_code_bytes(K, N));
    uint16_t* out = static_cast<uint16_t*>(w);
    if (f16) {
        if (has_zeros)
            dequant_ref_kernel<true, F16><<<grid, kPackThreads, 0, stream>>>(p, s, z, out, K, N);
        else
            dequant_ref_kernel<false, F16><<<grid, kPackThreads, 0, stream>>>(p, s, nullptr, out, K,
                                                                              N);
    } else if (has_zeros) {
        dequant_ref_kernel<true, Bf16><<<grid, kPackThreads, 0, stream>>>(p, s, z, out, K, N);
    } else {
        dequant_ref_kernel<false, Bf16><<<grid, kPackThreads, 0, stream>>>(p, s, nullptr, out, K, N);
    }
    return cudaGetLastError();
}

}  // namespace w4a16
