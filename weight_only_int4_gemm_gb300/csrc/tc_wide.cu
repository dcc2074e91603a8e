// tc_wide.cu -- W4A16 GEMM on the tcgen05 tensor cores for wide batches
// (more than 128 rows of x), with the dequantised weight tile in shared memory.
//
// "Give Me BF16 or Give Me Death" (summary), "Inference with W4A16": the
// 4-bit weights are rebuilt to 16-bit values inside the matrix
// multiplication and multiplied on 16-bit tensor cores with higher-precision
// accumulation; at large batch the layer is compute-bound.  "When
// quantization pays -- and when it does not" (model of a decode step): the
// dequantisation runs on the CUDA cores and is only free while another pipe is
// longer -- so here it runs in dedicated producer warps, overlapped with the
// asynchronous tensor pipe.
//
// At wide batches every MMA is long (N up to 256), so one issuing thread keeps
// the tensor pipe busy and the copies are large; this kernel keeps the simple
// single-issuer pipeline with the weight tile in shared memory.
//
// Tile (operands swapped so the weight tile is the 128-row MMA operand):
//   D[128 weight columns][bn batch rows] (fp32, TMEM)
//     += W^T[128][64 k] (bf16, smem, dequantised by producer warps)
//      . X^T[64 k][bn]  (bf16, smem, TMA from x[B][K])
// Persistent CTAs (one per SM) take work items (column tile, batch tile, K
// split) round robin and stream K in 64-row blocks through two rings: a ring
// of packed-code + x stages (as deep as shared memory allows, an even number
// of slots) and a ring of 4 dequantised weight tiles.  Warp roles:
//   warp 0      : TMA thread -- bulk-copies the packed codes of the block (one
//                 contiguous copy) and tensor-copies the x block (128-byte
//                 swizzle), one mbarrier with the expected byte count per slot;
//   warp 1      : TMEM allocator + the single MMA-issuing thread
//                 (tcgen05.mma kind::f16, 4 x K=16 per block, commit per slot
//                 to "empty" and per item to the accumulator's "full");
//   warps 2..17 : dequant producers, two groups of 8 warps taking alternate
//                 stages -- packed codes (smem) -> lop3 magic decode -> bf16
//                 (q - z) * s -> 128-byte-swizzled K-major rows of the weight
//                 tile; proxy fence; arrive;
//   warps 18..21: epilogue (tcgen05.ld 32 lanes x 16 columns -> bf16 y, or
//                 fp32 split-K reductions), one TMEM lane quadrant each.
// mbarrier waits test only the parity of a phase, so every waiter must wait
// for a barrier's uses in order: the groups take alternate stages, so the ring
// depth is even (a slot's consecutive uses fall to the same group) and the
// tile ring's depth (4) is too.
// Two TMEM accumulators alternate between items, so the epilogue of one item
// overlaps the main loop of the next.
// Every mbarrier wait is bounded; on expiry the kernel records
// W4A16_ERR_TIMEOUT in the device status word, drains and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "dequant.cuh"
#include "epilogue.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace w4a16 {
namespace {

using namespace ptx;

constexpr int kBlockK = 64;                  // K rows per pipeline stage
constexpr int kTileN = 128;                  // weight columns per tile (MMA M)
constexpr int kASlots = 4;                   // ring of dequantised weight tiles
constexpr int kMaxRawSlots = 32;             // ring of packed codes + x tiles
constexpr size_t kSmemBudget = 227 * 1024;
constexpr int kDequantWarp0 = 2;
constexpr int kDequantGroups = 2;            // groups of 8 warps take alternate stages
constexpr int kDequantWarps = 8;             // warps per group (one weight tile each)
constexpr int kEpilogueWarp0 = kDequantWarp0 + kDequantGroups * kDequantWarps;  // 18..21
constexpr int kNumWarps = kEpilogueWarp0 + 4;
constexpr int kThreads = 32 * kNumWarps;     // 704
constexpr uint32_t kATileBytes = kTileN * kBlockK * 2;   // 16 KB
constexpr uint32_t kRawBytes = kTileN * kBlockK / 2;     // 4 KB of packed codes
constexpr unsigned long long kTimeoutNs = 2000000000ull; // 2 s per wait

struct Args {
    const uint8_t* packed;
    const uint16_t* scales;
    const uint32_t* zeros;
    uint16_t* y;
    float* partial;      // fp32 accumulator [B][N], zero between calls (split > 1)
    uint32_t* counters;
    unsigned int* status;
    int B, K, N;
    int bn;             // MMA N (batch rows per tile), multiple of 16
    int kb_per_split;   // K blocks per split
    int split;
    int nkb;            // total K blocks (K / 64)
    int col_tiles, batch_tiles, items;
    uint32_t acc_cols;  // TMEM columns per accumulator (power of two >= max(32, bn))
    int raw_slots;      // depth of the codes + x ring
    int force_timeout;  // test hook: wait on a barrier nobody arrives at
    Epilogue epi;          // fused output epilogue (plain bf16 when mode == 0)
};

// ------------------------------------------------------------ kernel

struct SharedTail {
    uint64_t raw_full[kMaxRawSlots];   // TMA bytes landed (codes + x)
    uint64_t raw_empty[kMaxRawSlots];  // MMAs of the stage finished (commit)
    uint64_t a_full[kASlots];          // weight tile dequantised (8 warp arrivals)
    uint64_t a_empty[kASlots];         // MMAs reading the weight tile finished (commit)
    uint64_t tmem_full[2];             // accumulator complete (commit)
    uint64_t tmem_empty[2];            // accumulator drained by the epilogue (4 warps)
    uint64_t never;                    // test hook: nobody arrives here
    uint32_t tmem_base;
    int abort;
};

// Shared memory: [kASlots weight tiles of 16 KB][raw_slots x (x tile bn*128 B,
// packed codes 4 KB)][tail]; every operand tile starts on a 1024-byte boundary.
__host__ __device__ constexpr uint32_t raw_slot_bytes(int bn) {
    return (uint32_t)bn * kBlockK * 2 + kRawBytes;
}

struct Item {
    int col_tile, batch_tile, split_idx, n0, b0, nvalid, kb_begin, nkb;
};

__device__ __forceinline__ Item decode_item(const Args& a, int it) {
    Item t;
    t.col_tile = it % a.col_tiles;
    const int rest = it / a.col_tiles;
    t.batch_tile = rest % a.batch_tiles;
    t.split_idx = rest / a.batch_tiles;
    t.n0 = t.col_tile * kTileN;
    t.b0 = t.batch_tile * a.bn;
    t.nvalid = min(kTileN, a.N - t.n0);
    t.kb_begin = t.split_idx * a.kb_per_split;
    t.nkb = min(a.kb_per_split, a.nkb - t.kb_begin);
    return t;
}

__device__ __forceinline__ void epilogue_bar() {  // the 4 epilogue warps only
    asm volatile("bar.sync 2, 128;" ::: "memory");
}

template <bool kHasZeros, bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
wide_kernel(const __grid_constant__ CUtensorMap xmap, const Args a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled operand tiles
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int R = a.raw_slots;
    const uint32_t rbytes = raw_slot_bytes(a.bn);
    uint8_t* raw_base = smem + kASlots * kATileBytes;
    SharedTail* tail = reinterpret_cast<SharedTail*>(raw_base + R * rbytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = &tail->abort;

    auto a_tile = [&](int sa) { return smem + sa * kATileBytes; };
    auto x_tile = [&](int s) { return raw_base + s * rbytes; };
    auto raw_tile = [&](int s) { return raw_base + s * rbytes + a.bn * kBlockK * 2; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(smem_u32(&tail->raw_full[s]), 1);
            mbar_init(smem_u32(&tail->raw_empty[s]), 1);
        }
        for (int s = 0; s < kASlots; ++s) {
            mbar_init(smem_u32(&tail->a_full[s]), kDequantWarps);
            mbar_init(smem_u32(&tail->a_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tail->tmem_full[b]), 1);
            mbar_init(smem_u32(&tail->tmem_empty[b]), 4);
        }
        mbar_init(smem_u32(&tail->never), 1);
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
    // The next kernel on the stream may start now.  This one writes y and the
    // workspace, and reads x, only after the previous kernel has finished: the
    // TMA thread waits before its first x copy, and everything else is ordered
    // after that through mbarriers.  The packed codes do not depend on the
    // previous kernel, so the first stages' code copies go out before.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            const uint32_t xbytes = (uint32_t)a.bn * kBlockK * 2;
            const Item first = decode_item(a, blockIdx.x);
            const int pre = min(R, first.nkb);
            for (int i = 0; i < pre; ++i) {
                const uint32_t bar = smem_u32(&tail->raw_full[i]);
                const uint32_t cb = 2u * (uint32_t)first.nvalid * 16;  // two 32-row chunks
                mbar_arrive_expect_tx(bar, cb + xbytes);
                bulk_g2s(smem_u32(raw_tile(i)),
                         a.packed + packed_tile_base(a.K, first.col_tile) +
                             (size_t)(2 * (first.kb_begin + i)) * first.nvalid * 16,
                         cb, bar);
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            int stage = 0, issued = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x) {
                const Item t = decode_item(a, it);
                const uint32_t cb = 2u * (uint32_t)t.nvalid * 16;
                const uint8_t* tile_codes = a.packed + packed_tile_base(a.K, t.col_tile);
                for (int i = 0; i < t.nkb; ++i, ++stage) {
                    const int s = stage % R;
                    const uint32_t bar = smem_u32(&tail->raw_full[s]);
                    const int kb = t.kb_begin + i;
                    if (stage >= pre) {
                        if (stage >= R &&
                            !wait_bounded(smem_u32(&tail->raw_empty[s]), ((stage / R) - 1) & 1,
                                          abort, a.status, kTimeoutNs)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar, cb + xbytes);
                        bulk_g2s(smem_u32(raw_tile(s)), tile_codes + (size_t)(2 * kb) * t.nvalid * 16,
                                 cb, bar);
                    }
                    tma_load_2d(smem_u32(x_tile(s)), &xmap, kb * kBlockK, t.b0, bar);
                    issued = stage + 1;
                }
            }
            // After an expired wait, every copy in flight must land before the
            // CTA exits; stages whose code copy went out early still need their
            // x copy for the barrier to complete.
            if (!ok) {
                for (int i = issued; i < pre; ++i)
                    tma_load_2d(smem_u32(x_tile(i)), &xmap, (first.kb_begin + i) * kBlockK, first.b0,
                                smem_u32(&tail->raw_full[i]));
                const int last = max(issued, pre);
                for (int i = max(0, last - R); i < last; ++i)
                    wait_bounded(smem_u32(&tail->raw_full[i % R]), (i / R) & 1, abort, a.status,
                                 kTimeoutNs);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc_bf16(kTileN, a.bn);
            bool ok = true;
            if (a.force_timeout)
                ok = wait_bounded(smem_u32(&tail->never), 0, abort, a.status,
                                  (unsigned long long)a.force_timeout * 1000000ull);
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
                    const int s = stage % R;
                    const int sa = stage % kASlots;
                    if (!wait_fast(smem_u32(&tail->raw_full[s]), (stage / R) & 1, abort, a.status,
                                   kTimeoutNs) ||
                        !wait_fast(smem_u32(&tail->a_full[sa]), (stage / kASlots) & 1, abort,
                                   a.status, kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t abase = smem_u32(a_tile(sa));
                    const uint32_t xbase = smem_u32(x_tile(s));
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk)
                        mma_bf16_ss(tmem_d, smem_desc_sw128(abase + 32 * kk),
                                    smem_desc_sw128(xbase + 32 * kk), idesc, (i | kk) != 0);
                    mma_commit(smem_u32(&tail->a_empty[sa]));
                    mma_commit(smem_u32(&tail->raw_empty[s]));
                }
                mma_commit(smem_u32(&tail->tmem_full[acc]));  // fires once this item's MMAs are done
            }
            if (!ok) {
                // let the epilogue drain: both accumulators "complete" once
                // every issued MMA has finished
                mma_commit(smem_u32(&tail->tmem_full[0]));
                mma_commit(smem_u32(&tail->tmem_full[1]));
            }
        }
    } else if (warp < kEpilogueWarp0) {
        // ---------------- dequant producers (warps 2..17): two groups of 8 warps
        // take alternate stages, so two weight tiles are decoded at a time
        const int dw = warp - kDequantWarp0;
        const int grp = dw / kDequantWarps;                  // stage parity handled
        const int t256 = (dw % kDequantWarps) * 32 + lane;   // 0..255 within the group
        const int r = t256 & (kTileN - 1);                   // weight column within the tile
        const int h = t256 >> 7;                             // which 32-row chunk of the block
        int stage = 0;
        bool ok = true;
        for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x) {
            const Item t = decode_item(a, it);
            const int n = min(t.n0 + r, a.N - 1);
            for (int i = 0; i < t.nkb; ++i, ++stage) {
                if ((stage & 1) != grp) continue;
                const int s = stage % R;
                const int sa = stage % kASlots;
                const int g = (t.kb_begin + i) >> 1;  // two 64-row blocks per group of 128
                const uint32_t s2 = scale_pair(__ldg(a.scales + (size_t)g * a.N + n));
                const uint32_t z2 = kHasZeros ? zero_pair(load_zero(a.zeros, a.N, g, n))
                                              : kSymmetricZeroPair;
                bool landed = wait_fast(smem_u32(&tail->raw_full[s]), (stage / R) & 1, abort,
                                        a.status, kTimeoutNs);
                if (landed && stage >= kASlots)
                    landed = wait_fast(smem_u32(&tail->a_empty[sa]), ((stage / kASlots) - 1) & 1,
                                       abort, a.status, kTimeoutNs);
                if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform exit
                    ok = false;
                    break;
                }
                const uint4 q = reinterpret_cast<const uint4*>(raw_tile(s))[h * t.nvalid + min(r, t.nvalid - 1)];
                const uint32_t words[4] = {q.x, q.y, q.z, q.w};
                uint8_t* row = a_tile(sa) + r * 128;
#pragma unroll
                for (int jw = 0; jw < 4; ++jw) {
                    uint32_t p[4];
                    dequant_word(words[jw], z2, s2, p);
                    const int chunk = (4 * h + jw) ^ (r & 7);  // 128-byte swizzle
                    *reinterpret_cast<uint4*>(row + chunk * 16) = make_uint4(p[0], p[1], p[2], p[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tail->a_full[sa]));
            }
        }
    } else {
        // ---------------- epilogue (warps 10..13; TMEM lane quadrant = warp % 4)
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
                const int nn = t.n0 + quad * 32 + lane;
                const uint32_t taddr = tmem_base + acc * a.acc_cols + ((uint32_t)(quad * 32) << 16);
                for (int c0 = 0; c0 < a.bn; c0 += 16) {
                    float v[16];
                    tmem_ld_16(taddr + c0, v);
                    if (kFused && a.split == 1) {
                        // fused epilogue; b is the same in every lane (the
                        // SiLU form pairs lanes)
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int b = t.b0 + c0 + jj;
                            if (b < a.B) epi_store_lane_fused(a.y, a.N, b, nn, v[jj], nn < a.N, a.epi);
                        }
                    } else if (nn < a.N) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int b = t.b0 + c0 + jj;
                            if (b < a.B) {
                                if (a.split == 1)
                                    a.y[(size_t)b * a.N + nn] = (uint16_t)epi_f32_to_bf16(v[jj]);
                                else
                                    asm volatile("red.global.add.f32 [%0], %1;"
                                                 ::"l"(a.partial + (size_t)b * a.N + nn), "f"(v[jj])
                                                 : "memory");
                            }
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
                __shared__ int s_last;
                if (warp == kEpilogueWarp0 && lane == 0) {
                    uint32_t prev;
                    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                                 : "=r"(prev)
                                 : "l"(counter)
                                 : "memory");
                    s_last = (prev == (uint32_t)(a.split - 1));
                }
                epilogue_bar();
                if (s_last) {
                    __threadfence();
                    // 4 columns per thread and 8 loads in flight: the sums come
                    // back from L2, so latency, not bandwidth, sets the pace
                    const int rows = min(a.bn, a.B - t.b0);
                    const int c4n = t.nvalid / 4;
                    const int total = rows * c4n;
                    const int et = threadIdx.x - 32 * kEpilogueWarp0;
                    for (int e0 = et; e0 < total; e0 += 128 * 8) {
                        float4 v[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int e = e0 + 128 * j;
                            if (e < total) {
                                const int rr = e / c4n, cc = 4 * (e - (e / c4n) * c4n);
                                v[j] = __ldcg(reinterpret_cast<const float4*>(
                                    a.partial + (size_t)(t.b0 + rr) * a.N + t.n0 + cc));
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int e = e0 + 128 * j;
                            if (e < total) {
                                const int rr = e / c4n, cc = 4 * (e - (e / c4n) * c4n);
                                const size_t off = (size_t)(t.b0 + rr) * a.N + t.n0 + cc;
                                if constexpr (kFused)
                                    epi_store4_fused(a.y, a.N, t.b0 + rr, t.n0 + cc, v[j].x, v[j].y,
                                           v[j].z, v[j].w, a.epi);
                                else
                                    epi_store4_plain(a.y, a.N, t.b0 + rr, t.n0 + cc, v[j].x, v[j].y,
                                           v[j].z, v[j].w, a.epi);
                                __stcg(reinterpret_cast<float4*>(a.partial + off),
                                       make_float4(0.f, 0.f, 0.f, 0.f));
                            }
                        }
                    }
                    if (et == 0) *counter = 0u;
                }
                epilogue_bar();  // s_last is reused by the next item
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

// Even: the two dequant groups take alternate stages, so a slot's consecutive
// uses fall to the same group.
int raw_slots_for(int bn) {
    const size_t avail = kSmemBudget - 1024 - sizeof(SharedTail) - (size_t)kASlots * kATileBytes;
    return (int)std::min<size_t>(kMaxRawSlots, avail / raw_slot_bytes(bn)) & ~1;
}

size_t smem_bytes(int bn) {
    return (size_t)kASlots * kATileBytes + (size_t)raw_slots_for(bn) * raw_slot_bytes(bn) +
           sizeof(SharedTail) + 1024;
}

uint32_t acc_cols_for(int bn) {
    uint32_t c = 32;
    while (c < (uint32_t)bn) c <<= 1;
    return c;
}

}  // namespace

TcPlan plan_tc_wide(int B, int K, int N, int num_sms) {
    TcPlan p{};
    p.batch_tiles = (B + 255) / 256;
    const int per = (B + p.batch_tiles - 1) / p.batch_tiles;
    p.bn = std::min(256, (per + 15) / 16 * 16);
    p.col_tiles = (N + kTileN - 1) / kTileN;
    const int nkb = K / kBlockK;
    const long long tiles = (long long)p.col_tiles * p.batch_tiles;
    // persistent CTAs (one per SM) take items round robin; choose the K split
    // minimising the busiest CTA's K blocks plus a fixed cost per item and a
    // small cost per split (accumulator traffic)
    double best = 1e300;
    int best_split = 1, best_kbps = nkb;
    for (int split = 1; split <= std::min(16, nkb); ++split) {
        const int kbps = (nkb + split - 1) / split;
        if (split > 1 && (kbps < 8 || tiles > kMaxCounters)) break;
        const int s = (nkb + kbps - 1) / kbps;
        const long long items = tiles * s;
        const long long per_cta = (items + num_sms - 1) / num_sms;
        const double cost = (double)per_cta * (kbps + 4) * (1.0 + 0.02 * (s - 1));
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

static cudaError_t launch_wide_impl(const TcPlan& p, const void* x, const void* packed, const void* scales,
                           bool has_zeros, void* y, int B, int K, int N, void* workspace,
                           unsigned int* status, int force_timeout_ms, const Epilogue& epi,
                           cudaStream_t stream) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    CUtensorMap xmap;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)B};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBlockK, (cuuint32_t)p.bn};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    Args a;
    a.packed = static_cast<const uint8_t*>(packed);
    a.scales = static_cast<const uint16_t*>(scales);
    a.zeros = reinterpret_cast<const uint32_t*>(static_cast<const char*>(packed) +
                                                packed_code_bytes(K, N));
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
    a.raw_slots = raw_slots_for(p.bn);
    a.force_timeout = force_timeout_ms;
    a.epi = epi;

    const size_t smem = smem_bytes(p.bn);
    const bool fused = epi.mode != 0;
    const void* kern =
        has_zeros ? (fused ? reinterpret_cast<const void*>(wide_kernel<true, true>)
                           : reinterpret_cast<const void*>(wide_kernel<true, false>))
                  : (fused ? reinterpret_cast<const void*>(wide_kernel<false, true>)
                           : reinterpret_cast<const void*>(wide_kernel<false, false>));
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    void* args[] = {&xmap, &a};
    const int grid = std::min(a.items, p.grid);
    return launch_with_pdl(kern, dim3(grid), dim3(kThreads), smem, stream, args);
}

cudaError_t launch_tc_wide(const TcPlan& p, const void* x, const void* packed,
                           const void* scales, bool has_zeros, void* y, int B, int K, int N,
                           void* workspace, unsigned int* status, int force_timeout_ms,
                           const Epilogue& epi, cudaStream_t stream) {
    return launch_wide_impl(p, x, packed, scales, has_zeros, y, B, K, N, workspace, status,
                            force_timeout_ms, epi, stream);
}

}  // namespace w4a16
