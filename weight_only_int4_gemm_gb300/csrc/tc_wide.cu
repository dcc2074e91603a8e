// tc_wide.cu -- W4A16 GEMM on the tcgen05 tensor cores for batches of more
// than 16 rows of x: one or two MMA-issuing threads, the dequantised weight tile in
// tensor memory.
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
// Tile (operands swapped so the weight tile is the 128-row MMA operand):
//   D[128 weight columns][bn batch rows] (fp32, TMEM)
//     += W^T[128][64 k] (bf16, TMEM: lane = weight column, 32-bit column j =
//                        the k pair (2j, 2j+1), written by the dequant warps
//                        with tcgen05.st)
//      . X^T[64 k][bn]  (bf16, smem, TMA from x[B][K])
// The tile lives in tensor memory: through shared memory its store and its
// operand read would add a third to the shared-memory traffic of a block
// (the x copy, the tensor core's x reads, the code copies), and the shared
// memory goes to deeper rings instead.  A block is 128 rows of K (one scale
// group, 8 MMAs of K = 16): the MMA-issuing thread's per-block waits and
// commits cost about as much as 4 short MMAs, so longer blocks keep more of
// its time on MMAs.
// Persistent CTAs (one per SM) take work items (batch tile, column tile, K
// split; the batch tile varies fastest, so the batch tiles of one weight tile
// run side by side and its second reading comes from L2) round robin.  Three
// rings keep the tensor pipe fed:
//   * codes: one stage per block (its packed codes, 8 KB, one bulk copy; the
//     group's scale row and, for the asymmetric format, zero-point row, two
//     more bulk copies).  The weights come from HBM, so this ring runs
//     furthest ahead; the dequant warps read scales from it and never wait on
//     a global load;
//   * x: the block's activations per slot (two 2-D tensor copies of 64 K
//     rows, 128-byte swizzle, from L2);
//   * A: dequantised 128 x 128 weight tiles in TMEM, 64 columns each (4 to 8,
//     what the accumulators leave of the 512 columns).
// Warp roles:
//   warp 0      : code copies (one thread);
//   warp 1      : x copies (one thread);
//   warp 3      : TMEM allocator + MMA-issuing thread 0 (tcgen05.mma
//                 kind::f16, A from TMEM, 4 or 8 x K=16 per block);
//   warp 2      : MMA-issuing thread 1 at tiles of <= 128 rows (the two
//                 threads take alternate blocks into their own accumulators);
//   warps 4..7  : epilogue (tcgen05.ld, one TMEM lane quadrant each): the
//                 plain 16-bit output without a K split goes out as tensor
//                 stores of 16 x 32 chunks staged in shared memory, which run
//                 while the warp reads the next chunk (the accumulator is freed
//                 without waiting for y to reach memory; measured: gate_up
//                 4096 -> 28672 at B = 1024 170.0 -> 165.4 us); the fused
//                 epilogues go through a small transpose buffer so that every
//                 thread stores 16 bytes of y, and a K split's partial sums
//                 are added with one four-float vector reduction per thread;
//   warps 8..15 : dequant, two groups of four warps (one per TMEM lane
//                 quadrant) taking blocks in turn: each thread decodes the 128
//                 codes of its weight column (lop3 magic decode -> bf16
//                 (q - z) * s) and stores them to its TMEM lane.
// mbarrier waits test only the parity of a phase, so every waiter waits for a
// barrier's uses in order: block b uses code slot b mod RC, A slot b mod SA
// and x slot b mod SA (the x ring is as deep as the tile ring), both depths
// even, and the two dequant groups take alternate blocks, so every slot
// always serves one group; the MMA thread waits once per block (a block's
// tile is announced only once its x has landed too) and commits once: the
// commit frees the block's tile and its x slot together (the x copy thread
// waits on the tile ring's barriers).  Two TMEM
// accumulators alternate between items when TMEM has room for them
// (2 bn + 4 tiles <= 512 columns), so the epilogue of one item overlaps the
// main loop of the next.
// Every mbarrier wait is bounded; on expiry the kernel records
// W4A16_ERR_TIMEOUT in the device status word, drains and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "checks.cuh"
#include "dequant.cuh"
#include "epilogue.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace w4a16 {
namespace {

using namespace ptx;

constexpr int kGroupK = 128;                 // K rows per code stage (one scale group)
constexpr int kSubK = 64;                    // K rows per sub-block (4 MMAs of K = 16; one
                                             // 128-byte-swizzled x sub-tile, 32 TMEM columns)
constexpr int kTileN = 128;                  // weight columns per tile (MMA M)
constexpr int kMaxASlots = 8;                // ring of dequantised weight tiles (TMEM)
constexpr int kSubCols = kSubK / 2;          // TMEM columns per weight sub-tile (32)
constexpr int kTmemCols = 512;               // all of TMEM (one CTA per SM)
constexpr int kMaxCodeSlots = 16;            // ring of packed-code stages (128 rows each)
constexpr int kMaxXSlots = 16;               // ring of x blocks
constexpr size_t kSmemBudget = 227 * 1024;
constexpr int kCodeWarp = 0, kXWarp = 1, kMmaWarp = 3;  // warp 3: TMEM allocator, issuer 0
constexpr int kMmaWarp2 = 2;                 // issuer 1 (two issuers at tiles of <= 128 rows)
constexpr int kEpilogueWarp0 = 4;            // 4..7: TMEM lane quadrant = warp % 4
constexpr int kDequantWarp0 = 8;             // 8..15
constexpr int kDequantGroups = 2;            // groups of four warps take alternate blocks
constexpr int kDequantWarps = 4;             // one per TMEM lane quadrant
constexpr int kNumWarps = kDequantWarp0 + kDequantGroups * kDequantWarps;  // 16
constexpr int kThreads = 32 * kNumWarps;     // 512
constexpr uint32_t kStageCodeBytes = kTileN * kGroupK / 2;  // 8 KB: one group
constexpr uint32_t kScaleRowBytes = kTileN * 2;          // 256
constexpr uint32_t kZeroRowBytes = kTileN / 2;           // 64
constexpr uint32_t kCodeSlotBytes = kStageCodeBytes + kScaleRowBytes + kZeroRowBytes + 64;  // 8576
constexpr int kEpiRow = 36;                              // floats per transpose-buffer row (padded)
constexpr uint32_t kEpiBufBytes = 4 * 16 * kEpiRow * 4;  // 16 rows x 32 columns fp32 per warp
constexpr unsigned long long kTimeoutNs = 2000000000ull; // 2 s per wait

static_assert(kEpilogueWarp0 % 4 == 0 && kDequantWarp0 % 4 == 0,
              "TMEM lane quadrant of a warp is warp % 4");
static_assert(kCodeSlotBytes % 128 == 0, "code slots stay 128-byte aligned");
static_assert((16 * kEpiRow * 4) % 128 == 0 && 16 * kEpiRow * 4 >= 2 * 16 * 32 * 2,
              "a warp's transpose buffer holds two 128-byte aligned tensor-store chunks");

struct Args {
    const uint8_t* packed;
    const uint16_t* scales;
    const uint32_t* zeros;  // padded zero-point rows after the codes
    uint16_t* y;
    float* partial;      // fp32 accumulator [B][N], zero between calls (split > 1)
    uint32_t* counters;
    unsigned int* status;
    int B, K, N;
    int bn;             // MMA N (batch rows per tile), multiple of 16
    int gps;            // 128-row groups per K split
    int split;
    int ngroups;        // K / 128
    int col_tiles, batch_tiles, items;
    uint32_t acc_stride;  // TMEM columns per accumulator (bn rounded up to 32)
    int issuers;        // MMA-issuing threads (1 or 2), each with its own accumulator
    int bufs;           // accumulator sets alternating between items (1 or 2)
    int a_slots;        // dequantised tiles in TMEM (even, 4 .. 8)
    uint32_t a_col0;    // first TMEM column of the tile ring (after the accumulators)
    int code_slots, x_slots;
    uint32_t x_slot_bytes;
    uint32_t code_base, epi_base;  // shared-memory offsets (the x ring starts at 0)
    int zrow_words;     // words per padded zero-point row
    int force_timeout;  // test hook: wait on a barrier nobody arrives at
    Epilogue epi;       // fused output epilogue (plain bf16 when mode == 0)
    int y_tma;          // y written with tensor stores (plain output, no K split)
    const uint8_t* tag; // the packed blob's tag
    uint32_t tag_want[4];
    size_t code_bytes;  // packed codes (bounds checks)
};

// ------------------------------------------------------------ kernel

struct SharedTail {
    uint64_t code_full[kMaxCodeSlots];  // codes + scales (+ zero-points) of the stage landed
    uint64_t code_free[kMaxCodeSlots];  // read by every dequant warp
    uint64_t x_full[kMaxXSlots];        // x block landed
    uint64_t a_full[kMaxASlots];        // weight tile in TMEM and its x landed (one arrival
                                        // per warp of the dequant group)
    uint64_t a_free[kMaxASlots];        // MMAs reading the weight tile finished (commit)
    uint64_t tmem_full[2];              // accumulator complete (commit)
    uint64_t tmem_empty[2];             // accumulator drained by the epilogue (4 warps)
    uint64_t mma_done;                  // final drain of the issued MMAs
    uint64_t never;                     // test hook: nobody arrives here
    uint32_t tmem_base;
    int abort;
    int s_last;
};

struct Item {
    int col_tile, batch_tile, split_idx, n0, b0, nvalid, g_begin, ng;
};

__device__ __forceinline__ Item decode_item(const Args& a, int it) {
    Item t;
    t.batch_tile = it % a.batch_tiles;
    const int rest = it / a.batch_tiles;
    t.col_tile = rest % a.col_tiles;
    t.split_idx = rest / a.col_tiles;
    t.n0 = t.col_tile * kTileN;
    t.b0 = t.batch_tile * a.bn;
    t.nvalid = min(kTileN, a.N - t.n0);
    t.g_begin = t.split_idx * a.gps;
    t.ng = min(a.gps, a.ngroups - t.g_begin);
    return t;
}

// Ring position (slot, parity of the slot's current use), stepped without
// divisions.
struct Ring {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++s == n) {
            s = 0;
            ph ^= 1u;
        }
    }
};

__device__ __forceinline__ void epilogue_bar() {  // the 4 epilogue warps only
    asm volatile("bar.sync 2, 128;" ::: "memory");
}

// The packed codes, scale row and zero-point row of group g of item t.
template <bool kHasZeros>
__device__ __forceinline__ void issue_code_stage(const Args& a, const Item& t, int g,
                                                 uint8_t* slot, uint32_t bar) {
    const uint32_t cb = 4u * (uint32_t)t.nvalid * 16u;      // 4 chunks of 32 rows
    const uint32_t sb = (uint32_t)t.nvalid * 2u;            // multiple of 16 (N % 8 == 0)
    const uint32_t zb = kHasZeros ? (((uint32_t)t.nvalid / 2u + 15u) & ~15u) : 0u;
    const size_t off = packed_tile_base(a.K, t.col_tile) + (size_t)(4 * g) * t.nvalid * 16;
    const bool ok = in_bounds(off + cb <= a.code_bytes && g < a.ngroups &&
                                  t.n0 + t.nvalid <= a.N &&
                                  (!kHasZeros || (size_t)(t.n0 / 8) * 4 + zb <= (size_t)a.zrow_words * 4),
                              a.status);
    mbar_arrive_expect_tx(bar, ok ? cb + sb + zb : 0u);  // debug build: skip the copies
    if (!ok) return;
    bulk_g2s(smem_u32(slot), a.packed + off, cb, bar);
    bulk_g2s(smem_u32(slot + kStageCodeBytes), a.scales + (size_t)g * a.N + t.n0, sb, bar);
    if (kHasZeros)
        bulk_g2s(smem_u32(slot + kStageCodeBytes + kScaleRowBytes),
                 a.zeros + (size_t)g * a.zrow_words + t.n0 / 8, zb, bar);
}

// kSub: 64-row sub-blocks per block (1 or 2).  A block is the unit of the
// MMA thread's waits and commits and of the dequant groups' turns.
template <bool kHasZeros, bool kFused, int kSub, class Fmt>
__global__ void __launch_bounds__(kThreads, 1)
wide_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
            const Args a) {
    constexpr int kACols = kSubCols * kSub;         // TMEM columns per weight tile
    constexpr int kBlocksPerStage = 2 / kSub;       // blocks per code stage
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled x tiles
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int RC = a.code_slots;
    const int RX = a.x_slots;
    const int SA = a.a_slots;
    SharedTail* tail = reinterpret_cast<SharedTail*>(smem + a.epi_base + kEpiBufBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = &tail->abort;

    auto x_tile = [&](int s) { return smem + (size_t)s * a.x_slot_bytes; };
    auto code_slot = [&](int s) { return smem + a.code_base + (size_t)s * kCodeSlotBytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < RC; ++s) {
            mbar_init(smem_u32(&tail->code_full[s]), 1);
            // a stage is read by every group that has a block in it
            mbar_init(smem_u32(&tail->code_free[s]),
                      kDequantWarps * (kBlocksPerStage == 2 ? kDequantGroups : 1));
        }
        for (int s = 0; s < RX; ++s) {
            mbar_init(smem_u32(&tail->x_full[s]), 1);
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(smem_u32(&tail->a_full[s]), kDequantWarps);
            mbar_init(smem_u32(&tail->a_free[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tail->tmem_full[b]), a.issuers);  // one commit per issuer
            mbar_init(smem_u32(&tail->tmem_empty[b]), 4);
        }
        mbar_init(smem_u32(&tail->mma_done), a.issuers);
        mbar_init(smem_u32(&tail->never), 1);
        tail->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
        if (a.y_tma)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&ymap)) : "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tail->tmem_base)), "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tail->tmem_base;
    // The next kernel on the stream may start now.  This one reads x, and
    // writes y and the workspace, only after the previous kernel has finished:
    // the x thread waits before its first copy, and everything else that
    // touches x, y or the workspace is ordered after that through mbarriers.
    // The packed weights do not depend on the previous kernel (weights are
    // written by kernels that do not trigger early launches), so the code ring
    // starts filling at once.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kCodeWarp) {
        // ---------------- code stages: one per 128-row group
        if (lane == 0 && !blob_tag_matches(a.tag, a.tag_want))
            atomicExch(a.status, kStatusBadBlob);  // not a blob of this layout / shape
        if (lane == 0) {
            Ring q;
            int issued = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x) {
                const Item t = decode_item(a, it);
                for (int c = 0; c < t.ng; ++c, ++issued, q.next(RC)) {
                    if (issued >= RC &&
                        !wait_fast(smem_u32(&tail->code_free[q.s]), q.ph ^ 1u, abort, a.status,
                                   kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    issue_code_stage<kHasZeros>(a, t, t.g_begin + c, code_slot(q.s),
                                                smem_u32(&tail->code_full[q.s]));
                }
            }
            // After an expired wait, every copy in flight must land before the
            // CTA exits: wait for the latest use of every slot.
            if (!ok)
                for (int i = max(0, issued - RC); i < issued; ++i)
                    wait_bounded(smem_u32(&tail->code_full[i % RC]), (i / RC) & 1, abort,
                                 a.status, kTimeoutNs);
        }
    } else if (warp == kXWarp) {
        // ---------------- x blocks
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            Ring q;
            int issued = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x) {
                const Item t = decode_item(a, it);
                for (int i = 0; i < t.ng * kBlocksPerStage; ++i, ++issued, q.next(RX)) {
                    if (issued >= RX &&
                        !wait_fast(smem_u32(&tail->a_free[q.s]), q.ph ^ 1u, abort, a.status,
                                   kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_u32(&tail->x_full[q.s]);
                    mbar_arrive_expect_tx(bar, a.x_slot_bytes);
                    const int k0 = t.g_begin * kGroupK + i * kSub * kSubK;
#pragma unroll
                    for (int u = 0; u < kSub; ++u)
                        tma_load_2d(smem_u32(x_tile(q.s) + (uint32_t)u * (a.x_slot_bytes / kSub)),
                                    &xmap, k0 + u * kSubK, t.b0, bar);
                }
            }
            if (!ok)
                for (int i = max(0, issued - RX); i < issued; ++i)
                    wait_bounded(smem_u32(&tail->x_full[i % RX]), (i / RX) & 1, abort, a.status,
                                 kTimeoutNs);
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp2) {
        // ---------------- MMA issuers.  Issuer `me` takes the CTA's blocks b
        // with b % issuers == me -- with two issuers the same split as the
        // dequant groups' -- into its own accumulator (the epilogue adds
        // them): one thread issues a tcgen05.mma only every ~80 cycles at
        // tiles of <= 128 rows, below the tensor pipe's rate, so there two
        // threads issue.  A block's weight tile is announced only once its x
        // block has landed too (the dequant warps check it), so there is one
        // wait per block, made for the issuer's next block while this block's
        // last MMA is still to be issued: the tensor pipe's queue holds about
        // one MMA, and the wait would otherwise leave it idle.
        const int me = warp == kMmaWarp ? 0 : 1;
        const int I = a.issuers;
        if (lane == 0 && me < I) {
            const uint32_t idesc = instr_desc_f16kind(kTileN, a.bn, Fmt::kTcFormat);
            bool ok = true;
            if (a.force_timeout)
                ok = wait_bounded(smem_u32(&tail->never), 0, abort, a.status,
                                  (unsigned long long)a.force_timeout * 1000000ull);
            // descriptor of x slot 0; slot and K step add to its start-address
            // field (16-byte units, no carry out of it)
            const uint64_t xdesc0 = smem_desc_sw128(smem_u32(x_tile(0)));
            const uint32_t xslot16 = a.x_slot_bytes >> 4;
            const uint32_t a_tmem0 = tmem_base + a.a_col0;
            const uint32_t xsub16 = (uint32_t)a.bn * 8;  // one x sub-tile (bn x 128 B), 16-byte units
            // ring position of this issuer's next block: A slot = x slot = b % SA
            // (the two rings have one depth), stepped by I (SA is a multiple of I)
            int sl = me;
            uint32_t ph = 0;
            int gb0 = 0;  // CTA-wide index of the item's first block
            int j = 0;
            for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x, ++j) {
                const Item t = decode_item(a, it);
                const int acc = a.bufs == 2 ? (j & 1) : 0;
                const int use = a.bufs == 2 ? (j >> 1) : j;
                if (use >= 1 && !wait_bounded(smem_u32(&tail->tmem_empty[acc]), (use - 1) & 1,
                                              abort, a.status, kTimeoutNs)) {
                    ok = false;
                    break;
                }
                const uint32_t tmem_d =
                    tmem_base + (uint32_t)(acc * I + me) * a.acc_stride;
                const int nb = t.ng * kBlocksPerStage;
                int i = ((me - gb0) % I + I) % I;  // this issuer's first block of the item
                if (i < nb) {
                    if (!wait_test_first(smem_u32(&tail->a_full[sl]), ph, abort, a.status,
                                         kTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                for (bool first = true; i < nb; i += I, first = false) {
                    const uint32_t ta = a_tmem0 + (uint32_t)(sl * kACols);
                    const uint64_t xd = xdesc0 + (uint64_t)((uint32_t)sl * xslot16);
                    mma_bf16_ts(tmem_d, ta, xd, idesc, first ? 0u : 1u);
#pragma unroll
                    for (int kk = 1; kk < 4 * kSub - 1; ++kk)
                        mma_bf16_ts(tmem_d, ta + 8 * kk,
                                    xd + (uint64_t)((kk >> 2) * xsub16 + 2 * (kk & 3)), idesc, 1u);
                    const int done_slot = sl;
                    sl += I;
                    if (sl >= SA) {
                        sl -= SA;
                        ph ^= 1u;
                    }
                    if (i + I < nb) {
                        ok = wait_test_first(smem_u32(&tail->a_full[sl]), ph, abort, a.status,
                                             kTimeoutNs);
                        tc_fence_after();
                    }
                    mma_bf16_ts(tmem_d, ta + 8 * (4 * kSub - 1),
                                xd + (uint64_t)((kSub - 1) * xsub16 + 6), idesc, 1u);
                    // one commit per block releases both its weight tile and its x
                    // slot (the two rings have the same depth)
                    mma_commit(smem_u32(&tail->a_free[done_slot]));
                    if (!ok) break;
                }
                if (!ok) break;
                // fires once this issuer's MMAs of the item are done (it may
                // have none: then at once)
                mma_commit(smem_u32(&tail->tmem_full[acc]));
                gb0 += nb;
            }
            if (!ok) {
                // let the epilogue drain: both accumulators "complete" once
                // every issued MMA has finished
                mma_commit(smem_u32(&tail->tmem_full[0]));
                mma_commit(smem_u32(&tail->tmem_full[1]));
            }
            // every issued MMA has finished before TMEM is released, also after
            // an abort (issued MMAs wait on nothing, so this wait is short)
            mma_commit(smem_u32(&tail->mma_done));
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(&tail->mma_done), 0) && globaltimer() - t0 < kTimeoutNs) {
            }
        }
    } else if (warp >= kDequantWarp0) {
        // ---------------- dequant: group grp (four warps, one per TMEM lane
        // quadrant) takes blocks grp, grp + 2, ...: block b is 64 kSub-row
        // block b % kBlocksPerStage of code stage b / kBlocksPerStage, A slot
        // b % SA and x slot b % RX -- SA and RX are even, so every A and x slot
        // serves one group; with one block per stage RC is even too, and with
        // two each group reads every stage.  Each thread owns one weight
        // column = one TMEM lane and decodes its 64 kSub codes.
        const int grp = (warp - kDequantWarp0) / kDequantWarps;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // weight column within the tile
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16) + a.a_col0;
        constexpr int kCodeStep = kBlocksPerStage == 2 ? 1 : kDequantGroups;
        int cs = kBlocksPerStage == 2 ? 0 : grp;  // code slot of this group's current block
        int sa = grp, xs = grp;                   // its A and x slots
        uint32_t cph = 0, aph = 0, xph = 0;
        int own = 0;                       // blocks of this group so far
        int gb = 0;                        // blocks walked by the CTA
        bool ok = true;
        for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x) {
            const Item t = decode_item(a, it);
            const int rr = min(r, t.nvalid - 1);  // lanes past a ragged edge repeat a column
            for (int c = 0; c < t.ng * kBlocksPerStage; ++c, ++gb) {
                if ((gb & 1) != grp) continue;
                const int jb = kBlocksPerStage == 2 ? (c & 1) : 0;  // block within the stage
                bool landed = wait_fast(smem_u32(&tail->code_full[cs]), cph, abort, a.status,
                                        kTimeoutNs);
                // the tile slot is free once the MMAs of its previous block are done
                if (landed && gb >= SA)
                    landed = wait_fast(smem_u32(&tail->a_free[sa]), aph ^ 1u, abort, a.status,
                                       kTimeoutNs);
                if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform exit
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* slot = code_slot(cs);
                const uint32_t s2 = scale_pair(
                    reinterpret_cast<const uint16_t*>(slot + kStageCodeBytes)[rr]);
                uint32_t z2 = Fmt::kSymZero2;
                if (kHasZeros) {
                    const uint32_t zw = reinterpret_cast<const uint32_t*>(
                        slot + kStageCodeBytes + kScaleRowBytes)[rr >> 3];
                    z2 = zero_pair<Fmt>((zw >> (4 * (rr & 7))) & 0xFu);
                }
                const uint4* codes = reinterpret_cast<const uint4*>(slot) + (size_t)(2 * jb) * t.nvalid;
                // chunk h (rows 32h .. 32h+31 of the block) -> TMEM columns 16h .. 16h+15
                const uint32_t col = lane_addr + (uint32_t)(sa * kACols);
#pragma unroll
                for (int h = 0; h < 2 * kSub; ++h) {
                    // chunk 4g + 2jb + h of the group (swizzled run)
                    const uint4 qw = codes[h * t.nvalid + (rr ^ packed_swizzle(2 * jb + h))];
                    const uint32_t words[4] = {qw.x, qw.y, qw.z, qw.w};
                    uint32_t v[16];
#pragma unroll
                    for (int jw = 0; jw < 4; ++jw)
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp)
                            v[4 * jw + pp] = dequant_pair<Fmt>(words[jw], pp, z2, s2);
                    tmem_st_16(col + 16 * h, v);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                bool xok = true;
                if (lane == 0) {
                    mbar_arrive(smem_u32(&tail->code_free[cs]));  // this warp read the stage
                    // the tile is announced once the block's x has landed too
                    xok = wait_fast(smem_u32(&tail->x_full[xs]), xph, abort, a.status, kTimeoutNs);
                    if (xok) mbar_arrive(smem_u32(&tail->a_full[sa]));
                }
                cs += kCodeStep;
                if (cs >= RC) {
                    cs -= RC;
                    cph ^= 1u;
                }
                sa += kDequantGroups;
                if (sa >= SA) {
                    sa -= SA;
                    aph ^= 1u;
                }
                xs += kDequantGroups;
                if (xs >= RX) {
                    xs -= RX;
                    xph ^= 1u;
                }
                ++own;
                if (!__shfl_sync(0xffffffffu, xok ? 1 : 0, 0)) {  // warp-uniform exit
                    ok = false;
                    break;
                }
            }
        }
    } else if (warp >= kEpilogueWarp0 && warp < kEpilogueWarp0 + 4) {
        // ---------------- epilogue (warps 4..7; TMEM lane quadrant = warp % 4)
        const int quad = warp & 3;
        float* buf = reinterpret_cast<float*>(smem + a.epi_base) + quad * 16 * kEpiRow;
        // tensor-store staging: two 16 x 32 16-bit chunks in the warp's buffer
        // (128-byte aligned: the buffer is 2304 bytes per warp)
        uint16_t* stage = reinterpret_cast<uint16_t*>(buf);
        int sbuf = 0;
        const int I = a.issuers;
        int j = 0;
        int gb0 = 0;  // CTA-wide index of the item's first block
        for (int it = blockIdx.x; it < a.items; it += gridDim.x, ++j) {
            const Item t = decode_item(a, it);
            const int acc = a.bufs == 2 ? (j & 1) : 0;
            const int use = a.bufs == 2 ? (j >> 1) : j;
            // accumulators holding sums: issuer k's, if it had a block of this item
            const int nb = t.ng * kBlocksPerStage;
            const bool has0 = I == 1 || nb >= 2 || (gb0 & 1) == 0;
            const bool has1 = I == 2 && (nb >= 2 || (gb0 & 1) == 1);
            gb0 += nb;
            const bool done = wait_bounded(smem_u32(&tail->tmem_full[acc]), use & 1, abort,
                                           a.status, kTimeoutNs);
            tc_fence_after();
            const bool live = __all_sync(0xffffffffu, done && !*abort);
            if (live) {  // tcgen05.ld is warp-collective
                const int nq = t.n0 + quad * 32;  // this warp's 32 columns
                const uint32_t taddr = tmem_base + (uint32_t)(acc * I) * a.acc_stride +
                                       ((uint32_t)(quad * 32) << 16);
                for (int c0 = 0; c0 < a.bn; c0 += 16) {
                    float v[16];
                    tmem_ld_16(taddr + (has0 ? 0u : a.acc_stride) + c0, v);
                    if (has0 && has1) {
                        float v1[16];
                        tmem_ld_16(taddr + a.acc_stride + c0, v1);
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] += v1[i];
                    }
                    if (!kFused && a.y_tma) {
                        // rows c0 .. c0 + 15 of the tile, this warp's 32 columns, as
                        // 16-bit values in the staging chunk, then one tensor store
                        // that runs while the next chunk is read: the epilogue does
                        // not wait for y to reach memory before it frees the
                        // accumulator.  The chunk's previous store must have read it.
                        if (lane == 0) bulk_wait_read_1();
                        __syncwarp();
                        uint16_t* st = stage + sbuf * 512;
#pragma unroll
                        for (int i = 0; i < 16; ++i) st[i * 32 + lane] = (uint16_t)Fmt::from_f32(v[i]);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&ymap, smem_u32(st), nq, t.b0 + c0);
                            bulk_commit_group();
                        }
                        sbuf ^= 1;
                        continue;
                    }
                    // transpose through shared memory: row i of the chunk, 32 columns
#pragma unroll
                    for (int i = 0; i < 16; ++i) buf[i * kEpiRow + lane] = v[i];
                    __syncwarp();
                    if (a.split == 1) {
                        // 8 consecutive columns of one row per thread
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const int i = 8 * rr + (lane >> 2);
                            const int c8 = 8 * (lane & 3);
                            const int b = t.b0 + c0 + i;
                            const int n = nq + c8;
                            const float4 lo = *reinterpret_cast<const float4*>(buf + i * kEpiRow + c8);
                            const float4 hi =
                                *reinterpret_cast<const float4*>(buf + i * kEpiRow + c8 + 4);
                            if (b < a.B && n < a.N && in_bounds(n + 8 <= a.N, a.status)) {
                                if constexpr (kFused) {
                                    epi_store4_fused(a.y, a.N, b, n, lo.x, lo.y, lo.z, lo.w, a.epi);
                                    epi_store4_fused(a.y, a.N, b, n + 4, hi.x, hi.y, hi.z, hi.w, a.epi);
                                } else {
                                    *reinterpret_cast<uint4*>(a.y + (size_t)b * a.N + n) = make_uint4(
                                        Fmt::from_f32(lo.x) | (Fmt::from_f32(lo.y) << 16),
                                        Fmt::from_f32(lo.z) | (Fmt::from_f32(lo.w) << 16),
                                        Fmt::from_f32(hi.x) | (Fmt::from_f32(hi.y) << 16),
                                        Fmt::from_f32(hi.z) | (Fmt::from_f32(hi.w) << 16));
                                }
                            }
                        }
                    } else {
                        // 4 consecutive columns of one row per thread: one vector reduction
#pragma unroll
                        for (int rr = 0; rr < 4; ++rr) {
                            const int i = 4 * rr + (lane >> 3);
                            const int c4 = 4 * (lane & 7);
                            const int b = t.b0 + c0 + i;
                            const int n = nq + c4;
                            const float4 p = *reinterpret_cast<const float4*>(buf + i * kEpiRow + c4);
                            if (b < a.B && n < a.N && in_bounds(n + 4 <= a.N, a.status))
                                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                                             ::"l"(a.partial + (size_t)b * a.N + n), "f"(p.x),
                                             "f"(p.y), "f"(p.z), "f"(p.w)
                                             : "memory");
                        }
                    }
                    __syncwarp();  // the buffer is rewritten by the next chunk
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
                if (!in_bounds((size_t)t.batch_tile * a.col_tiles + t.col_tile < (size_t)kMaxCounters,
                               a.status))
                    counter = a.counters;  // debug build: a valid word (the sum is then wrong)
                if (warp == kEpilogueWarp0 && lane == 0) {
                    uint32_t prev;
                    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                                 : "=r"(prev)
                                 : "l"(counter)
                                 : "memory");
                    tail->s_last = (prev == (uint32_t)(a.split - 1));
                }
                epilogue_bar();
                if (tail->s_last) {
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
                        for (int jj = 0; jj < 8; ++jj) {
                            const int e = e0 + 128 * jj;
                            if (e < total) {
                                const int rr = e / c4n, cc = 4 * (e - rr * c4n);
                                if (in_bounds(t.b0 + rr < a.B && t.n0 + cc + 4 <= a.N, a.status))
                                    v[jj] = __ldcg(reinterpret_cast<const float4*>(
                                        a.partial + (size_t)(t.b0 + rr) * a.N + t.n0 + cc));
                            }
                        }
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const int e = e0 + 128 * jj;
                            if (e < total) {
                                const int rr = e / c4n, cc = 4 * (e - rr * c4n);
                                const size_t off = (size_t)(t.b0 + rr) * a.N + t.n0 + cc;
                                if (t.b0 + rr >= a.B || t.n0 + cc + 4 > a.N) continue;
                                if constexpr (kFused)
                                    epi_store4_fused(a.y, a.N, t.b0 + rr, t.n0 + cc, v[jj].x,
                                                     v[jj].y, v[jj].z, v[jj].w, a.epi);
                                else
                                    epi_store4_plain<Fmt>(a.y, a.N, t.b0 + rr, t.n0 + cc, v[jj].x,
                                                     v[jj].y, v[jj].z, v[jj].w, a.epi);
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
        // y's tensor stores complete before the CTA exits (their source is
        // this CTA's shared memory)
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
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

// 64-row sub-blocks per block: two (longer blocks, half the MMA thread's
// per-block waits and commits per MMA) up to 160 batch rows; one at wider
// tiles, where the x slots of twice-as-long blocks leave too shallow a ring.
// Measured over the decode shapes: at bn = 144, 128-row blocks take gate_up
// 4096 -> 28672 at B = 270 from 74.7 to 62.7 us; from bn = 176 on they are
// 10-40 % slower.
int sub_blocks(int bn) { return bn <= 160 ? 2 : 1; }

// Shared memory: [x ring][code ring][epilogue buffer][tail] (+ 1 KB of
// alignment slack).  Six code stages (the weights come from HBM), then as
// many x slots as fit (an even 2 .. 8: x comes from L2), then the rest to the
// code ring (an even number).
struct WideLayout {
    int x_slots, code_slots;
    uint32_t x_slot_bytes, code_base, epi_base;
    size_t smem;
};

WideLayout wide_layout(int bn, int sub) {
    WideLayout l;
    // kSub sub-tiles of bn x 128 B, each a multiple of 1024 (bn % 8 == 0)
    l.x_slot_bytes = (uint32_t)bn * kSubK * 2 * (uint32_t)sub;
    const size_t fixed = 1024 + kEpiBufBytes + sizeof(SharedTail);
    const size_t avail = kSmemBudget - fixed;
    const size_t want_code = 6 * (size_t)kCodeSlotBytes;
    int xs = avail > want_code ? (int)((avail - want_code) / l.x_slot_bytes) : 0;
    xs = std::max(2, std::min(8, xs)) & ~1;  // even: a slot serves one dequant group
    const size_t left = avail > (size_t)xs * l.x_slot_bytes ? avail - (size_t)xs * l.x_slot_bytes : 0;
    l.code_slots = (int)std::min<size_t>(kMaxCodeSlots, left / kCodeSlotBytes) & ~1;  // even
    l.x_slots = xs;
    l.code_base = (uint32_t)xs * l.x_slot_bytes;
    l.epi_base = l.code_base + (uint32_t)l.code_slots * kCodeSlotBytes;
    l.smem = 1024 + (size_t)l.epi_base + kEpiBufBytes + sizeof(SharedTail);
    return l;
}

// TMEM: [accumulator set 0][set 1, when both fit with 4 tile slots][tiles]; a
// set holds one accumulator per MMA-issuing thread (two at tiles of <= 128
// rows, where one thread cannot issue MMAs as fast as the pipe runs them:
// ~80 cycles per MMA from one thread, ~40-60 per MMA per SM from two or three
// -- measured with a separate microbenchmark at N = 64).
struct TmemLayout {
    uint32_t acc_stride, a_col0;
    int issuers, bufs, a_slots;
};

TmemLayout tmem_layout(int bn, int sub) {
    TmemLayout t;
    const uint32_t acols = (uint32_t)(kSubCols * sub);
    t.acc_stride = (uint32_t)((bn + 31) / 32 * 32);
    t.issuers = bn <= 128 ? 2 : 1;
    const uint32_t set = (uint32_t)t.issuers * t.acc_stride;  // one accumulator per issuer
    t.bufs = 2 * set + 4 * acols <= (uint32_t)kTmemCols ? 2 : 1;
    t.a_col0 = (uint32_t)t.bufs * set;
    t.a_slots = std::min(kMaxASlots, (int)((kTmemCols - t.a_col0) / acols)) & ~1;
    return t;
}

}  // namespace

// Work decomposition for batches above 16 rows.  A work item is one
// 128-column tile of W for one batch tile of bn rows, over a range of whole
// 128-row groups of K; persistent CTAs (one per SM) take items round robin,
// so the time is that of the busiest CTA: ceil(items / SMs) items.  Every
// weight tile is decoded once per batch tile, so smaller batch tiles cost
// dequantisation, larger ones leave SMs idle; a K split adds the partial
// sums' reductions.  The cost of an item, in SM cycles, is a non-negative
// least-squares fit (relative errors) to the measured times of the decode
// shapes (qkv 4096 -> 6144, o_proj 4096 -> 4096, gate_up 4096 -> 28672,
// down 14336 -> 4096, lm_head 4096 -> 128256 at B = 32 .. 1024, every batch
// tile count in range and K split; median error 5 %), whose picks cost 0.7 %
// more than the fastest measured plans over the decode step:
//   per 64 rows of K:  bn <= 160 (128-row blocks): 302 + 1.5 bn cycles (the
//                      issuing threads' per-block waits and commit, not the
//                      MMAs, set the pace);  wider (64-row blocks): 332 + 2.0 bn;
//   per item with a K split: 82 bn more, the reductions of its bn x 128
//                      partial sums.
// The search stays inside the range the fit was made on -- the smallest
// batch-tile count and the two above it, K splits of 1 to 4 -- where the
// fit is checked against measurements; outside it the fit extrapolates.
TcPlan plan_tc_wide(int B, int K, int N, int num_sms) {
    TcPlan best{};
    double best_cost = 1e300;
    const int G = K / kGroup;
    const int col_tiles = (N + kTileN - 1) / kTileN;
    const int min_bt = (B + 255) / 256;
    for (int bt = min_bt; bt <= min_bt + 2; ++bt) {
        const int per = (B + bt - 1) / bt;
        const int bn = std::min(256, (per + 15) / 16 * 16);
        if (bn < 32 && bt > min_bt) break;
        const int batch_tiles = (B + bn - 1) / bn;
        const long long tiles = (long long)col_tiles * batch_tiles;
        const double rows64 = sub_blocks(bn) == 2 ? 302.1 + 1.5 * bn : 332.3 + 2.0 * bn;
        for (int split = 1; split <= std::min(4, G); ++split) {
            const int gps = (G + split - 1) / split;
            const int s = (G + gps - 1) / gps;  // no empty splits
            if (s != split) continue;
            // no K split beside tiles wider than 160 rows: their bn x 128
            // reductions cost more than the fit expects (down 14336 -> 4096
            // at B = 384: 59.8 us with bn = 192 and two splits, 55.7 us with
            // bn = 128 and three)
            if (s > 1 && bn > 160) break;
            if (s > 1 && tiles > kMaxCounters - 2) break;
            const long long items = tiles * s;
            const long long per_cta = (items + num_sms - 1) / num_sms;
            const double reduce = s > 1 ? 82.4 * bn : 0.0;
            const double cost = (double)per_cta * (2.0 * gps * rows64 + reduce);
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best.bn = bn;
                best.batch_tiles = batch_tiles;
                best.split = s;
                best.kb_per_split = 2 * gps;
                best.sub = sub_blocks(bn);
            }
        }
    }
    best.col_tiles = col_tiles;
    best.grid = (int)std::min<long long>((long long)col_tiles * best.batch_tiles * best.split,
                                         num_sms);
    best.wide = true;
    return best;
}

PlanResources wide_resources(const TcPlan& p, int B, int N) {
    (void)B;
    (void)N;
    PlanResources r{};
    const WideLayout lay = wide_layout(p.bn, p.sub);
    const TmemLayout tm = tmem_layout(p.bn, p.sub);
    r.smem = lay.smem;
    r.ctas_per_sm = 1;
    r.issuers = tm.issuers;
    r.acc_bufs = tm.bufs;
    // as launched: the x ring as deep as the tile ring
    r.tile_slots = std::min(tm.a_slots, lay.x_slots);
    r.x_slots = r.tile_slots;
    r.code_slots = lay.code_slots;
    r.tmem_cols = (int)tm.a_col0 + r.tile_slots * kSubCols * p.sub;
    r.block_rows = kSubK * p.sub;
    return r;
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
    const cuuint32_t box[2] = {(cuuint32_t)kSubK, (cuuint32_t)p.bn};  // 128-byte rows (swizzle span)
    const cuuint32_t estr[2] = {1, 1};
    // (bf16 or fp16 x: the copy moves 16-bit patterns, one map type serves both)
    if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // y for the tensor-store epilogue: boxes of 16 rows x 32 columns (64-byte
    // rows, unswizzled), used for the plain 16-bit output without a K split
    // when y is at least one box in each dimension (a box may then overhang
    // the tensor's edge, whose elements the store skips; a box larger than
    // the whole tensor is not used); otherwise, or if the encoder refuses (an
    // unaligned y), the epilogue stores per thread
    CUtensorMap ymap;
    bool y_tma = false;
    if (epi.mode == 0 && p.split == 1 && N >= 32 && B >= 16) {
        const cuuint64_t ydims[2] = {(cuuint64_t)N, (cuuint64_t)B};
        const cuuint64_t ystrides[1] = {(cuuint64_t)N * 2};
        const cuuint32_t ybox[2] = {32, 16};
        y_tma = enc(&ymap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y, ydims, ystrides, ybox, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    if (!y_tma) ymap = xmap;  // unused

    const WideLayout lay = wide_layout(p.bn, p.sub);
    const TmemLayout tm = tmem_layout(p.bn, p.sub);
    if (lay.x_slots < 2 || (lay.x_slots & 1) || lay.code_slots < 2 || lay.smem > kSmemBudget ||
        tm.a_slots < 4)
        return cudaErrorInvalidConfiguration;
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
    a.gps = p.kb_per_split / 2;
    a.split = p.split;
    a.ngroups = K / kGroup;
    a.col_tiles = p.col_tiles;
    a.batch_tiles = p.batch_tiles;
    a.items = p.col_tiles * p.batch_tiles * p.split;
    a.acc_stride = tm.acc_stride;
    a.issuers = tm.issuers;
    a.bufs = tm.bufs;
    // The x ring and the weight-tile ring have one depth: block b's single
    // commit then frees A slot b % SA and x slot b % SA together (a commit
    // costs the MMA thread about as much as an MMA; measured: one commit per
    // block instead of two, gate_up 4096 -> 28672 at B = 1024 183 -> 169 us).
    a.a_slots = std::min(tm.a_slots, lay.x_slots);
    a.a_col0 = tm.a_col0;
    a.code_slots = lay.code_slots;
    a.x_slots = a.a_slots;
    a.x_slot_bytes = lay.x_slot_bytes;
    a.code_base = lay.code_base;
    a.epi_base = lay.epi_base;
    a.zrow_words = packed_zero_row_words(N);
    a.force_timeout = force_timeout_ms;
    a.epi = epi;
    a.y_tma = y_tma ? 1 : 0;
    a.tag = a.packed + packed_tag_offset(K, N, has_zeros);
    a.code_bytes = code_bound_bytes(K, N);
    {
        const BlobTag want = blob_tag(K, N, has_zeros);
        for (int i = 0; i < 4; ++i) a.tag_want[i] = want.w[i];
    }

    const size_t smem = lay.smem;
    const bool fused = epi.mode != 0;
    const void* kern = nullptr;
    if (epi.f16) {
        switch ((p.sub == 2 ? 2 : 0) + (has_zeros ? 1 : 0)) {
            case 0: kern = reinterpret_cast<const void*>(wide_kernel<false, false, 1, F16>); break;
            case 1: kern = reinterpret_cast<const void*>(wide_kernel<true, false, 1, F16>); break;
            case 2: kern = reinterpret_cast<const void*>(wide_kernel<false, false, 2, F16>); break;
            default: kern = reinterpret_cast<const void*>(wide_kernel<true, false, 2, F16>); break;
        }
    } else {
        switch ((p.sub == 2 ? 4 : 0) + (has_zeros ? 2 : 0) + (fused ? 1 : 0)) {
            case 0: kern = reinterpret_cast<const void*>(wide_kernel<false, false, 1, Bf16>); break;
            case 1: kern = reinterpret_cast<const void*>(wide_kernel<false, true, 1, Bf16>); break;
            case 2: kern = reinterpret_cast<const void*>(wide_kernel<true, false, 1, Bf16>); break;
            case 3: kern = reinterpret_cast<const void*>(wide_kernel<true, true, 1, Bf16>); break;
            case 4: kern = reinterpret_cast<const void*>(wide_kernel<false, false, 2, Bf16>); break;
            case 5: kern = reinterpret_cast<const void*>(wide_kernel<false, true, 2, Bf16>); break;
            case 6: kern = reinterpret_cast<const void*>(wide_kernel<true, false, 2, Bf16>); break;
            default: kern = reinterpret_cast<const void*>(wide_kernel<true, true, 2, Bf16>); break;
        }
    }
    cudaError_t err =
        set_smem_limit(kern, smem);
    if (err != cudaSuccess) return err;
    void* args[] = {&xmap, &ymap, &a};
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
