// dequant.cuh -- packed weight layout and the register-level INT4 -> bf16
// decode shared by every kernel of the library (GEMMs and dequant_ref).
//
// Decode ("When quantization pays -- and when it does not", section
// "Counting c from the kernel, not from intuition"): OR-ing a 4-bit code q
// into the low fraction bits of bf16 128.0 (0x4300) gives exactly bf16(128+q);
// subtracting bf16(128+z) (z = 8 for the symmetric format, i.e. 136.0 =
// 0x4308) gives the exact integer q - z; one round-to-nearest-even bf16
// multiply by the group scale then gives w = RNE_bf16((q - z) * s).  One
// lop3 builds two such values at once, one in each 16-bit half.
//
// Packed layout (version W4A16_PACKED_LAYOUT = 4):
//   codes: the N columns are cut into tiles of 128 (the last tile holds
//   w = N - 128*t columns when N is not a multiple of 128).  Tile t starts at
//   byte 64*K*t; inside it, chunk c (rows 32c .. 32c+31) is w consecutive
//   16-byte entries, one per column, so every (tile, run of chunks) is one
//   contiguous block -- a single bulk copy.  Column n's entry of chunk c sits
//   at position n XOR 2*(c mod 4) of the run (w is a multiple of 8, so the
//   swizzle stays inside the run): a warp whose eight-lane phases read four
//   chunks of two columns each then touches eight different bank groups of
//   shared memory instead of two.  The 16 bytes of (chunk c, column n) hold
//   the 32 codes of rows 32c .. 32c+31 of column n; word j holds rows
//   32c + 8j .. 32c + 8j + 7.  Inside a word, the codes of rows
//   (2i, 2i+1) (offsets within the word) sit in nibbles i and i + 4, i.e. in
//   the low and high 16-bit halves at the same bit offset 4i, so
//        (word >> 4i) & 0x000F000F  ==  { code(2i), code(2i+1) }.
//   zeros (asymmetric format only): the canonical uint32 [K/128][N/8] words,
//   after the codes, one group per row, each row padded with zero words to a
//   multiple of 4 words (16 bytes), so the zero-points of any 128-column tile
//   of a group are one 16-byte-aligned block a bulk copy can fetch.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "fmt16.cuh"

namespace w4a16 {

constexpr int kPackTileCols = 128;

// Width of column tile t.
__host__ __device__ inline int packed_tile_width(int N, int t) {
    return N - kPackTileCols * t < kPackTileCols ? N - kPackTileCols * t : kPackTileCols;
}

// Byte offset of tile t's block of codes.
__host__ __device__ inline size_t packed_tile_base(int K, int t) {
    return (size_t)64 * (size_t)K * (size_t)t;
}

// Swizzle of chunk c's run: column n of the tile sits at position n ^ swizzle.
__host__ __device__ constexpr int packed_swizzle(int c) { return 2 * (c & 3); }

// Index, in 16-byte units, of (chunk c, column n).
__host__ __device__ inline size_t packed_index16(int K, int N, int c, int n) {
    const int t = n / kPackTileCols;
    return packed_tile_base(K, t) / 16 + (size_t)c * packed_tile_width(N, t) +
           (size_t)((n - kPackTileCols * t) ^ packed_swizzle(c));
}

// Nibble position of row offset r (0..7) inside a packed word.
__host__ __device__ constexpr int packed_nibble_of_row(int r) {
    return (r & 1) ? 4 + (r >> 1) : (r >> 1);
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    // (a & b) | c, as one LOP3 (lookup table 0xF0 & 0xCC | 0xAA = 0xEA).
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// (P + z) in both halves (P = 128 for bf16, 1024 for fp16, fmt16.cuh): the
// value subtracted after the magic OR.
template <class Fmt = Bf16>
__device__ __forceinline__ uint32_t zero_pair(uint32_t z) {
    return Fmt::kMagic2 | (z * 0x00010001u);
}
constexpr uint32_t kSymmetricZeroPair = Bf16::kSymZero2;  // bf16 136.0 = 128 + 8, twice

// Scale broadcast to both halves.
__device__ __forceinline__ uint32_t scale_pair(uint16_t s) {
    return (uint32_t)s * 0x00010001u;
}

// Pair i (0..3) of a packed word: rows (2i, 2i+1) as two 16-bit values,
// exact RNE((q - z) * s) in each half (bf16 or fp16).
template <class Fmt = Bf16>
__device__ __forceinline__ uint32_t dequant_pair(uint32_t word, int i, uint32_t zero2,
                                                 uint32_t scale2) {
    const uint32_t magic = lop3_and_or(word >> (4 * i), 0x000F000Fu, Fmt::kMagic2);
    return Fmt::mul2(Fmt::sub2(magic, zero2), scale2);
}

// Pair i (0..3) of a packed word as the exact integers (q - z): the magic OR
// and the exact subtraction, without the scale.  Kernels that apply the group
// scale to an fp32 sum over the group use this.
template <class Fmt = Bf16>
__device__ __forceinline__ uint32_t code_pair(uint32_t word, int i, uint32_t zero2) {
    return Fmt::sub2(lop3_and_or(word >> (4 * i), 0x000F000Fu, Fmt::kMagic2), zero2);
}

// All 8 rows of a packed word, out[i] = rows (2i, 2i+1).
template <class Fmt = Bf16>
__device__ __forceinline__ void dequant_word(uint32_t word, uint32_t zero2, uint32_t scale2,
                                             uint32_t out[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = dequant_pair<Fmt>(word, i, zero2, scale2);
}

// Device check of a packed blob's tag (see launch.cuh): one 16-byte load.
__device__ __forceinline__ bool blob_tag_matches(const uint8_t* tag, const uint32_t (&want)[4]) {
    const uint4 t = *reinterpret_cast<const uint4*>(tag);
    return t.x == want[0] && t.y == want[1] && t.z == want[2] && t.w == want[3];
}

// Words per group row of the packed zero-points (N/8 rounded up to 4).
__host__ __device__ inline int packed_zero_row_words(int N) { return ((N >> 3) + 3) & ~3; }

// Zero-point nibble of column n, group g, from the packed zero-points.
__device__ __forceinline__ uint32_t load_zero(const uint32_t* zeros, int N, int g, int n) {
    const uint32_t w = __ldg(zeros + (size_t)g * packed_zero_row_words(N) + (n >> 3));
    return (w >> (4 * (n & 7))) & 0xFu;
}

}  // namespace w4a16
