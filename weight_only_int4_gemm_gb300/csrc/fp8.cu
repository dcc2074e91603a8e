// fp8.cu -- the W8A8-FP8 comparison path: dynamic per-token activation
// quantisation, per-output-channel weight quantisation, and the FP8 GEMM on
// the tcgen05 tensor cores.
//
// "Give Me BF16 or Give Me Death" (summary page), section "W8A8-FP
// Quantization: 8-Bit Floating-Point Weights and Activations": weights get one
// scale per output channel, activations one scale per token computed on the
// fly, s = max|v| / q_max, codes = nearest FP8 value of v / s; the product
// runs on FP8 tensor cores.  "When quantization pays -- and when it does
// not" (the three regimes): the 8-bit weight stream halves bf16's memory term
// and the FP8 tensor rate halves its math term, which is the comparison this
// path measures against W4A16.
//
// Format: E4M3 (no infinities, largest finite 448).  Quotients are binary32
// divisions, rounded once to E4M3 by the hardware conversion (nearest, ties
// to even, saturating); an all-zero row has scale 0 and codes 0.
//
// Weight layout for the GEMM (w8a8_fp8_pack_weight): the [N][K] codes are cut
// into tiles of 128 output channels x 128 k, each stored as one contiguous
// 16 KB block that is already the shared-memory image the MMA reads (rows of
// 128 bytes, 128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r & 7));
// tile t, k block kb sits at block t * (K / 128) + kb; channels past N are
// zero.  One bulk copy per stage then streams the weights: reading the [N][K]
// matrix as 2-D boxes of 128 rows x 128 bytes, K bytes apart, reached only
// about half the HBM bandwidth.
//
// GEMM tile (operands swapped so the weight tile is the 128-row MMA operand):
//   D[128 weight columns][bn batch rows] (fp32, TMEM)
//     += Wq[128 columns][128 k] (E4M3, smem, bulk copy) . Xq[bn rows][128 k]^T (TMA)
// Both operand tiles are 128 bytes per row, so they use the same K-major
// 128-byte-swizzled layout as the bf16 kernels' 64-element blocks; one stage
// is four tcgen05.mma kind::f8f6f4 (K = 32 each).  Persistent CTAs take work
// items (column tile, batch tile, K split) round robin.  Warp roles:
//   warp 0     : copy thread (weight block + activation tile per stage, one
//                mbarrier with the expected byte count);
//   warp 1     : TMEM allocator + the MMA-issuing thread (commit per stage to
//                "empty", per item to the accumulator's "full");
//   warps 2..5 : epilogue -- tcgen05.ld, y = acc * s_x[row] * s_w[column] ->
//                bf16, or fp32 split-K reductions and a final conversion by
//                the last CTA of a tile.
// Every mbarrier wait is bounded; on expiry the kernel records
// W4A16_ERR_TIMEOUT in the device status word, drains and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "launch.cuh"
#include "tc_ptx.cuh"

namespace w4a16 {
namespace {

using namespace ptx;

constexpr float kE4M3Max = 448.0f;

// ------------------------------------------------------------ quantisers

// Two binary32 values -> two E4M3 codes (nearest, ties to even, saturating):
// `lo` in the low byte, `hi` in the high byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Codes of eight consecutive bf16 values (one 16-byte load) with scale s > 0.
__device__ __forceinline__ uint2 encode8(uint4 v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        p[j] = cvt_e4m3x2(__fdiv_rn(bf16_lo(w[j]), s), __fdiv_rn(bf16_hi(w[j]), s));
    return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

constexpr int kRowThreads = 256;

// One CTA per row of x [B][K]: max |x| over the row, s = max / 448, codes.
__global__ void __launch_bounds__(kRowThreads)
fp8_quant_rows_kernel(const uint16_t* __restrict__ x, int K, uint8_t* __restrict__ xq,
                      float* __restrict__ sx) {
    const int b = blockIdx.x;
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)b * K);
    const int nv = K / 8;
    // launched with programmatic dependent launch: x comes from the previous
    // kernel, and the GEMM that follows may start its weight copies early
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float m = 0.0f;
    for (int i = threadIdx.x; i < nv; i += kRowThreads) {
        const uint4 v = __ldg(row + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float red[kRowThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0.0f;
#pragma unroll
    for (int i = 0; i < kRowThreads / 32; ++i) m = fmaxf(m, red[i]);
    const float s = __fdiv_rn(m, kE4M3Max);
    if (threadIdx.x == 0) sx[b] = s;
    uint2* out = reinterpret_cast<uint2*>(xq + (size_t)b * K);
    for (int i = threadIdx.x; i < nv; i += kRowThreads)
        out[i] = s > 0.0f ? encode8(__ldg(row + i), s) : make_uint2(0u, 0u);
}

constexpr int kColThreads = 128;

// Per output channel of W [K][N]: s_w[n] = max_k |W[k][n]| / 448.
__global__ void __launch_bounds__(kColThreads)
fp8_col_scale_kernel(const uint16_t* __restrict__ w, int K, int N, float* __restrict__ sw) {
    const int n = blockIdx.x * kColThreads + threadIdx.x;
    if (n >= N) return;
    float m = 0.0f;
    for (int k = 0; k < K; ++k)
        m = fmaxf(m, fabsf(__uint_as_float((uint32_t)__ldg(w + (size_t)k * N + n) << 16)));
    sw[n] = __fdiv_rn(m, kE4M3Max);
}

// Codes of 16 consecutive k of one channel, written as one 16-byte row piece
// of Wq [N][K] (the transposed, K-major layout the GEMM's TMA reads).
__global__ void __launch_bounds__(kColThreads)
fp8_quant_cols_kernel(const uint16_t* __restrict__ w, int K, int N, const float* __restrict__ sw,
                      uint8_t* __restrict__ wq) {
    const int n = blockIdx.x * kColThreads + threadIdx.x;
    const int k0 = blockIdx.y * 16;
    if (n >= N) return;
    const float s = sw[n];
    uint32_t p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float lo = __uint_as_float((uint32_t)__ldg(w + (size_t)(k0 + 2 * j) * N + n) << 16);
        const float hi =
            __uint_as_float((uint32_t)__ldg(w + (size_t)(k0 + 2 * j + 1) * N + n) << 16);
        p[j] = s > 0.0f ? cvt_e4m3x2(__fdiv_rn(lo, s), __fdiv_rn(hi, s)) : 0u;
    }
    *reinterpret_cast<uint4*>(wq + (size_t)n * K + k0) =
        make_uint4(p[0] | (p[1] << 16), p[2] | (p[3] << 16), p[4] | (p[5] << 16),
                   p[6] | (p[7] << 16));
}

constexpr int kPackThreads = 256;

// [N][K] codes -> tiled, pre-swizzled blocks (one thread per 16-byte chunk).
__global__ void __launch_bounds__(kPackThreads)
fp8_pack_kernel(const uint8_t* __restrict__ wq, int K, int N, uint8_t* __restrict__ packed,
                long long chunks) {
    const long long i = (long long)blockIdx.x * kPackThreads + threadIdx.x;
    if (i >= chunks) return;
    const int c = (int)(i & 7);               // 16-byte chunk of the 128-byte row
    const int r = (int)((i >> 3) & 127);      // channel inside the tile
    const long long blk = i >> 10;            // (tile, k block)
    const int nkb = K / 128;
    const int t = (int)(blk / nkb), kb = (int)(blk % nkb);
    const int n = t * 128 + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < N) v = *reinterpret_cast<const uint4*>(wq + (size_t)n * K + (size_t)kb * 128 + 16 * c);
    *reinterpret_cast<uint4*>(packed + (size_t)blk * 16384 + r * 128 + ((c ^ (r & 7)) * 16)) = v;
}

// ------------------------------------------------------------ GEMM

constexpr int kBlockK = 128;                          // k per stage (bytes per operand row)
constexpr int kTileN = 128;                           // weight columns per tile (MMA M)
constexpr uint32_t kWTileBytes = kTileN * kBlockK;    // 16 KB
constexpr int kMaxStages = 16;
constexpr int kEpilogueWarp0 = 2;
constexpr int kThreads = 32 * (kEpilogueWarp0 + 4);   // 192
constexpr size_t kSmemBudget = 227 * 1024;
constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per wait

struct Args {
    const uint8_t* wpacked;  // tiled weight blocks (fp8_pack_kernel)
    const float* sx;
    const float* sw;
    uint16_t* y;
    float* partial;      // fp32 accumulator [B][N], zero between calls (split > 1)
    uint32_t* counters;
    unsigned int* status;
    int B, K, N;
    int bn;              // MMA N (batch rows per tile), multiple of 16
    int kb_per_split, split, nkb;
    int col_tiles, batch_tiles, items;
    uint32_t acc_cols;   // TMEM columns per accumulator (power of two >= max(32, bn))
    int stages;          // depth of the operand ring
};

struct Tail {
    uint64_t full[kMaxStages];    // both operand tiles landed
    uint64_t empty[kMaxStages];   // the stage's MMAs finished (commit)
    uint64_t tmem_full[2];        // accumulator complete (commit)
    uint64_t tmem_empty[2];       // accumulator drained by the 4 epilogue warps
    uint32_t tmem_base;
    int abort;
    int last;                     // this CTA converts the tile (split-K)
};

__host__ __device__ constexpr uint32_t stage_bytes(int bn) {
    return kWTileBytes + (uint32_t)bn * kBlockK;
}

struct Item {
    int col_tile, batch_tile, n0, b0, kb_begin, nkb;
};

__device__ __forceinline__ Item decode_item(const Args& a, int it) {
    Item t;
    t.col_tile = it % a.col_tiles;
    const int rest = it / a.col_tiles;
    t.batch_tile = rest % a.batch_tiles;
    const int split_idx = rest / a.batch_tiles;
    t.n0 = t.col_tile * kTileN;
    t.b0 = t.batch_tile * a.bn;
    t.kb_begin = split_idx * a.kb_per_split;
    t.nkb = min(a.kb_per_split, a.nkb - t.kb_begin);
    return t;
}

__device__ __forceinline__ void epilogue_bar() {  // the 4 epilogue warps only
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int S = a.stages;
    const uint32_t sbytes = stage_bytes(a.bn);
    Tail* tail = reinterpret_cast<Tail*>(smem + S * sbytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = &tail->abort;
    auto w_tile = [&](int s) { return smem + s * sbytes; };
    auto w_block = [&](const Item& t, int kb) {
        return a.wpacked + ((size_t)t.col_tile * a.nkb + kb) * kWTileBytes;
    };
    auto x_tile = [&](int s) { return smem + s * sbytes + kWTileBytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&tail->full[s]), 1);
            mbar_init(smem_u32(&tail->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tail->tmem_full[b]), 1);
            mbar_init(smem_u32(&tail->tmem_empty[b]), 4);
        }
        tail->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tail->tmem_base)), "r"(2 * a.acc_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tail->tmem_base;
    // The next kernel on the stream may start now.  Activations, their scales,
    // y and the workspace are touched only after the previous kernel has
    // finished (the TMA thread waits before its first activation copy and
    // everything else follows it through mbarriers); the weights do not depend
    // on the previous kernel, so the first stages' weight copies go out before.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            const uint32_t xbytes = (uint32_t)a.bn * kBlockK;
            const uint64_t evict_first = l2_evict_first_policy();  // weights are read once
            const Item first = decode_item(a, blockIdx.x);
            const int pre = min(S, first.nkb);
            for (int i = 0; i < pre; ++i) {
                const uint32_t bar = smem_u32(&tail->full[i]);
                mbar_arrive_expect_tx(bar, kWTileBytes + xbytes);
                bulk_g2s_hint(smem_u32(w_tile(i)), w_block(first, first.kb_begin + i), kWTileBytes,
                              bar, evict_first);
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            int stage = 0, issued = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x) {
                const Item t = decode_item(a, it);
                for (int i = 0; i < t.nkb; ++i, ++stage) {
                    const int s = stage % S;
                    const uint32_t bar = smem_u32(&tail->full[s]);
                    const int kb = t.kb_begin + i;
                    if (stage >= pre) {
                        if (stage >= S &&
                            !wait_bounded(smem_u32(&tail->empty[s]), ((stage / S) - 1) & 1, abort,
                                          a.status, kTimeoutNs)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar, kWTileBytes + xbytes);
                        bulk_g2s_hint(smem_u32(w_tile(s)), w_block(t, kb), kWTileBytes, bar,
                                      evict_first);
                    }
                    tma_load_2d(smem_u32(x_tile(s)), &xmap, kb * kBlockK, t.b0, bar);
                    issued = stage + 1;
                }
            }
            // After an expired wait every copy in flight must land before the
            // CTA exits; stages whose weight copy went out early still need
            // their activation copy for the barrier to complete.
            if (!ok) {
                for (int i = issued; i < pre; ++i)
                    tma_load_2d(smem_u32(x_tile(i)), &xmap, (first.kb_begin + i) * kBlockK, first.b0,
                                smem_u32(&tail->full[i]));
                const int last = max(issued, pre);
                for (int i = max(0, last - S); i < last; ++i)
                    wait_bounded(smem_u32(&tail->full[i % S]), (i / S) & 1, abort, a.status,
                                 kTimeoutNs);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc_e4m3(kTileN, a.bn);
            bool ok = true;
            int stage = 0, j = 0;
            for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x, ++j) {
                const Item t = decode_item(a, it);
                const int acc = j & 1;
                if (j >= 2 && !wait_bounded(smem_u32(&tail->tmem_empty[acc]), ((j >> 1) - 1) & 1,
                                            abort, a.status, kTimeoutNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tmem_d = tmem_base + acc * a.acc_cols;
                for (int i = 0; i < t.nkb; ++i, ++stage) {
                    const int s = stage % S;
                    if (!wait_fast(smem_u32(&tail->full[s]), (stage / S) & 1, abort, a.status,
                                   kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t wbase = smem_u32(w_tile(s));
                    const uint32_t xbase = smem_u32(x_tile(s));
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 32; ++kk)
                        mma_f8_ss(tmem_d, smem_desc_sw128(wbase + 32 * kk),
                                  smem_desc_sw128(xbase + 32 * kk), idesc, (i | kk) != 0);
                    mma_commit(smem_u32(&tail->empty[s]));
                }
                mma_commit(smem_u32(&tail->tmem_full[acc]));
            }
            if (!ok) {
                // let the epilogue drain: both accumulators "complete" once
                // every issued MMA has finished
                mma_commit(smem_u32(&tail->tmem_full[0]));
                mma_commit(smem_u32(&tail->tmem_full[1]));
            }
        }
    } else {
        // ---------------- epilogue (TMEM lane quadrant = warp % 4)
        const int quad = warp & 3;
        int j = 0;
        for (int it = blockIdx.x; it < a.items; it += gridDim.x, ++j) {
            const Item t = decode_item(a, it);
            const int acc = j & 1;
            const bool done = wait_bounded(smem_u32(&tail->tmem_full[acc]), (j >> 1) & 1, abort,
                                           a.status, kTimeoutNs);
            tc_fence_after();
            const bool live = __all_sync(0xffffffffu, done && !*abort);
            if (live) {  // tcgen05.ld is warp-collective
                const int n = t.n0 + quad * 32 + lane;
                const bool col_ok = n < a.N;
                const float s_w = col_ok ? __ldg(a.sw + n) : 0.0f;
                const uint32_t taddr = tmem_base + acc * a.acc_cols + ((uint32_t)(quad * 32) << 16);
                for (int c0 = 0; c0 < a.bn; c0 += 16) {
                    float v[16];
                    tmem_ld_16(taddr + c0, v);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int b = t.b0 + c0 + jj;
                        if (b < a.B && col_ok) {
                            const float r = __fmul_rn(__fmul_rn(v[jj], __ldg(a.sx + b)), s_w);
                            if (a.split == 1)
                                a.y[(size_t)b * a.N + n] = f32_to_bf16_rn(r);
                            else
                                asm volatile("red.global.add.f32 [%0], %1;"
                                             ::"l"(a.partial + (size_t)b * a.N + n), "f"(r)
                                             : "memory");
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tail->tmem_empty[acc]));
            if (!live) break;
            if (a.split > 1) {
                // the last CTA of this tile to arrive converts the fp32 sum to
                // bf16 and clears the accumulator for the next call
                __threadfence();
                epilogue_bar();
                uint32_t* counter = a.counters + (size_t)t.batch_tile * a.col_tiles + t.col_tile;
                if (warp == kEpilogueWarp0 && lane == 0) {
                    uint32_t prev;
                    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                                 : "=r"(prev)
                                 : "l"(counter)
                                 : "memory");
                    tail->last = (prev == (uint32_t)(a.split - 1));
                }
                epilogue_bar();
                if (tail->last) {
                    __threadfence();
                    const int rows = min(a.bn, a.B - t.b0);
                    const int c4n = min(kTileN, a.N - t.n0) / 4;
                    const int total = rows * c4n;
                    const int et = threadIdx.x - 32 * kEpilogueWarp0;
                    for (int e = et; e < total; e += 128) {
                        const int rr = e / c4n, cc = 4 * (e - rr * c4n);
                        const size_t off = (size_t)(t.b0 + rr) * a.N + t.n0 + cc;
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.partial + off));
                        const uint32_t lo = (uint32_t)f32_to_bf16_rn(v.x) |
                                            ((uint32_t)f32_to_bf16_rn(v.y) << 16);
                        const uint32_t hi = (uint32_t)f32_to_bf16_rn(v.z) |
                                            ((uint32_t)f32_to_bf16_rn(v.w) << 16);
                        *reinterpret_cast<uint2*>(a.y + off) = make_uint2(lo, hi);
                        __stcg(reinterpret_cast<float4*>(a.partial + off),
                               make_float4(0.f, 0.f, 0.f, 0.f));
                    }
                    if (et == 0) *counter = 0u;
                }
                epilogue_bar();  // tail->last is reused by the next item
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(2 * a.acc_cols)
                     : "memory");
    }
}

// ------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major uint8 matrix [rows][K] read in boxes of 128 k x box_rows rows,
// 128-byte swizzle (the K-major operand layout of the MMA).
bool encode_operand(EncodeTiledFn enc, CUtensorMap* map, const void* base, int K, int rows,
                    int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {(cuuint32_t)kBlockK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Up to 128 batch rows two CTAs share an SM (two independent copy / MMA /
// epilogue pipelines, each with half the shared memory; measured on the
// linear set: B = 1 56.4 -> 50.7 us for the GEMMs, B = 64 127.6 -> 112.9 us and
// B = 128 198.6 -> 175.0 us per step); 256-row tiles run one CTA per SM.
int ctas_per_sm(int bn) { return bn <= 128 ? 2 : 1; }

int stages_for(int bn) {
    const size_t budget = ctas_per_sm(bn) == 2 ? kSmemBudget / 2 : kSmemBudget;
    const size_t avail = budget - 1024 - sizeof(Tail);
    return (int)std::min<size_t>(kMaxStages, avail / stage_bytes(bn));
}

size_t smem_bytes(int bn) {
    return (size_t)stages_for(bn) * stage_bytes(bn) + sizeof(Tail) + 1024;
}

uint32_t acc_cols_for(int bn) {
    uint32_t c = 32;
    while (c < (uint32_t)bn) c <<= 1;
    return c;
}

}  // namespace

Fp8Plan plan_fp8(int B, int K, int N, int num_sms_in) {
    Fp8Plan p{};
    p.batch_tiles = (B + 255) / 256;
    const int per = (B + p.batch_tiles - 1) / p.batch_tiles;
    p.bn = std::min(256, (per + 15) / 16 * 16);
    const int num_sms = num_sms_in * ctas_per_sm(p.bn);  // resident CTAs
    p.col_tiles = (N + kTileN - 1) / kTileN;
    const int nkb = K / kBlockK;
    const long long tiles = (long long)p.col_tiles * p.batch_tiles;
    // persistent CTAs (one per SM) take items round robin.  One SM streams
    // only a share of the HBM bandwidth, so the step time follows the busiest
    // CTA's stages (plus a fixed cost per item and, with a K split, the fp32
    // reduction of a bn x 128 tile: bn / 32 stage-equivalents), scaled up
    // when fewer items than SMs leave SMs idle
    double best = 1e300;
    int best_split = 1, best_kbps = nkb;
    for (int split = 1; split <= std::min(32, nkb); ++split) {
        const int kbps = (nkb + split - 1) / split;
        if (split > 1 && (kbps < 4 || tiles > kMaxCounters - 2)) break;
        const int s = (nkb + kbps - 1) / kbps;
        const long long items = tiles * s;
        const long long per_cta = (items + num_sms - 1) / num_sms;
        const double idle = items < num_sms ? (double)num_sms / (double)items : 1.0;
        const double cost =
            (double)per_cta * (kbps + 2 + (s > 1 ? p.bn / 32.0 : 0.0)) * idle;
        if (cost < best - 1e-9) {
            best = cost;
            best_split = s;
            best_kbps = kbps;
        }
    }
    p.split = best_split;
    p.kb_per_split = best_kbps;
    p.grid = (int)std::min<long long>(tiles * p.split, num_sms);
    return p;
}

size_t fp8_workspace_bytes(const Fp8Plan& p, int B, int N) {
    return p.split > 1 ? kCounterBytes + (size_t)B * N * sizeof(float) : 0;
}

cudaError_t launch_fp8_quantize_rows(const void* x, int B, int K, void* xq, float* sx,
                                     cudaStream_t stream) {
    const uint16_t* xp = static_cast<const uint16_t*>(x);
    uint8_t* xqp = static_cast<uint8_t*>(xq);
    void* args[] = {&xp, &K, &xqp, &sx};
    return launch_with_pdl(reinterpret_cast<const void*>(fp8_quant_rows_kernel), dim3(B),
                           dim3(kRowThreads), 0, stream, args);
}

cudaError_t launch_fp8_quantize_cols(const void* w, int K, int N, void* wq, float* sw,
                                     cudaStream_t stream) {
    const int cb = (N + kColThreads - 1) / kColThreads;
    fp8_col_scale_kernel<<<cb, kColThreads, 0, stream>>>(static_cast<const uint16_t*>(w), K, N, sw);
    fp8_quant_cols_kernel<<<dim3(cb, K / 16), kColThreads, 0, stream>>>(
        static_cast<const uint16_t*>(w), K, N, sw, static_cast<uint8_t*>(wq));
    return cudaGetLastError();
}

size_t fp8_packed_bytes(int K, int N) {
    return (size_t)((N + kTileN - 1) / kTileN) * kTileN * (size_t)K;
}

cudaError_t launch_fp8_pack(const void* wq, int K, int N, void* packed, cudaStream_t stream) {
    const long long chunks = (long long)fp8_packed_bytes(K, N) / 16;
    const long long blocks = (chunks + kPackThreads - 1) / kPackThreads;
    fp8_pack_kernel<<<(unsigned)blocks, kPackThreads, 0, stream>>>(
        static_cast<const uint8_t*>(wq), K, N, static_cast<uint8_t*>(packed), chunks);
    return cudaGetLastError();
}

cudaError_t launch_fp8_gemm(const Fp8Plan& p, const void* xq, const float* sx,
                            const void* wpacked, const float* sw, void* y, int B, int K, int N,
                            void* workspace, unsigned int* status, cudaStream_t stream) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    CUtensorMap xmap;
    if (!encode_operand(enc, &xmap, xq, K, B, p.bn)) return cudaErrorInvalidValue;
    Args a;
    a.wpacked = static_cast<const uint8_t*>(wpacked);
    a.sx = sx;
    a.sw = sw;
    a.y = static_cast<uint16_t*>(y);
    a.partial = ws_partials(workspace);
    a.counters = ws_counters(workspace);
    a.status = status;
    a.B = B;
    a.K = K;
    a.N = N;
    a.bn = p.bn;
    a.kb_per_split = p.kb_per_split;
    a.split = p.split;
    a.nkb = K / kBlockK;
    a.col_tiles = p.col_tiles;
    a.batch_tiles = p.batch_tiles;
    a.items = p.col_tiles * p.batch_tiles * p.split;
    a.acc_cols = acc_cols_for(p.bn);
    a.stages = stages_for(p.bn);
    const size_t smem = smem_bytes(p.bn);
    const void* kern = reinterpret_cast<const void*>(fp8_gemm_kernel);
    cudaError_t err =
        set_smem_limit(kern, smem);
    if (err != cudaSuccess) return err;
    void* args[] = {&xmap, &a};
    return launch_with_pdl(kern, dim3(std::min(a.items, p.grid)), dim3(kThreads), smem, stream,
                           args);
}

}  // namespace w4a16
