// tc_gemm.cu -- W4A16 GEMM on the 5th-generation tensor cores (tcgen05 MMA,
// TMA-fed activations), with the dequantised weight tile held in tensor memory.
//
// "Give Me BF16 or Give Me Death" (summary), "Inference with W4A16": the
// 4-bit weights are rebuilt to 16-bit values inside the matrix
// multiplication and multiplied on 16-bit tensor cores with higher-precision
// accumulation.  "When quantization pays -- and when it does not" (model of a
// decode step): the dequantisation runs on the CUDA cores and is only free
// while another pipe is longer -- so here it runs in dedicated warps,
// overlapped with the asynchronous copy and tensor pipes.
//
// Tile (operands swapped so the weight tile is the 128-row MMA operand):
//   D[128 weight columns][bn batch rows] (fp32, TMEM)
//     += W^T[128][64 k] (bf16, TMEM: lane = weight column, 32-bit column j =
//                        the k pair (2j, 2j+1), even k in the low half)
//      . X^T[64 k][bn]  (bf16, smem, 128-byte swizzle, TMA from x[B][K])
// The weight operand never touches shared memory: each dequant thread owns
// one weight column (one TMEM lane), decodes its 64 codes of a block into 32
// bf16 pairs and writes them with two tcgen05.st.
//
// Copies: a TMA operation costs a few hundred cycles of the SM's copy engine
// whatever its size, so the K loop is fed in copy stages of nsub 64-row blocks
// (nsub = 4 at small bn: 16 KB of packed codes per stage), each stage one bulk
// copy of codes, one tensor copy of the group scales (and one of the
// zero-points) and one 3-D tensor copy of all its x blocks; two producer
// threads take the stages in turn.  Codes and x travel in two rings: a code
// slot is free as soon as the dequant warps have read it, an x slot once the
// stage's MMAs finished, so the HBM stream of codes is not held up by the
// (slow to issue) MMAs.  Dequantisation and MMAs stay per 64-row block,
// through a ring of weight tiles in TMEM.
//
// Persistent CTAs (one per SM) take work items (column tile, batch tile, K
// split) round robin.  Up to four MMA-issuing threads take the 64-row blocks
// in turn, each into its own accumulator: MMAs issued by one thread run one
// after another, so at small bn (short MMAs) several issuers keep the tensor
// pipe busy; the epilogue adds the accumulators.  Warp roles:
//   warps 0, 25     : TMA producers (copy stages alternate between them);
//   warps 1-3, 24   : MMA issuers 0-3 (warp 1 also allocates TMEM);
//   warps 4-7       : epilogue, TMEM lane quadrant = warp % 4;
//   warps 8-23      : dequant, four groups of four warps taking 64-row blocks
//                     in turn; warp % 4 is the TMEM lane quadrant it writes.
// Every role keeps its ring positions as counters stepped once per stage: a
// role runs on one thread, where a division's dependent chain would cost as
// much as a stage's MMAs.  Accumulators are double-buffered between items when
// TMEM has room, so the epilogue of one item overlaps the main loop of the
// next.  Every mbarrier wait is bounded; on expiry the kernel records
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

constexpr int kBlockK = 64;                  // K rows per block (4 MMAs of K = 16)
constexpr int kTileN = 128;                  // weight columns per tile (MMA M)
constexpr int kMaxCodeSlots = 16;            // ring of packed codes + scales + zero-points
constexpr int kMaxXSlots = 16;               // ring of x tiles
constexpr int kMaxASlots = 12;               // ring of weight tiles in TMEM
constexpr int kTmemCols = 512;               // the whole of TMEM (one CTA per SM)
constexpr int kACols = kBlockK / 2;          // TMEM columns per weight tile
constexpr int kMaxIssuers = 4;
// Wider batches go to tc_wide.cu: measured on the Llama-3-8B decode step
// (129 GEMMs), the single-issuer wide-batch kernel is faster from 17 rows on
// (B = 24 / 32 / 48 / 64: 2655 / 2714 / 2903 / 3046 us per step against
// 2801 / 2897 / 3566 / 3969 us here).  This kernel serves the tensor-core path
// when it is forced at 16 rows or fewer.
constexpr int kMaxTmemBatch = 16;
constexpr int kEpilogueWarp0 = 4;            // 4..7
constexpr int kDequantWarp0 = 8;             // 8..23
constexpr int kDequantGroups = 4;            // groups of 4 warps (one per quadrant)
constexpr int kIssuer3Warp = kDequantWarp0 + 4 * kDequantGroups;  // 24
constexpr int kProducer1Warp = kIssuer3Warp + 1;                  // 25
constexpr int kNumWarps = kProducer1Warp + 1;
constexpr int kThreads = 32 * kNumWarps;     // 832
constexpr size_t kSmemBudget = 227 * 1024;
constexpr uint32_t kCodeBlockBytes = kTileN * kBlockK / 2;  // 4 KB of codes per block
constexpr uint32_t kScaleRowBytes = kTileN * 2;             // one group's scales of a tile
constexpr uint32_t kZeroRowBytes = kTileN / 2;              // one group's zero-points
constexpr unsigned long long kTimeoutNs = 2000000000ull;    // 2 s per wait

static_assert(kDequantWarp0 % 4 == 0 && kEpilogueWarp0 % 4 == 0,
              "TMEM lane quadrant of a warp is warp % 4");

struct Args {
    const uint8_t* packed;
    uint16_t* y;
    float* partial;        // fp32 accumulator [B][N], zero between calls (split > 1)
    uint32_t* counters;
    unsigned int* status;
    int B, K, N;
    int bn;                // MMA N (batch rows per tile), multiple of 16
    int nsub;              // 64-row blocks per copy stage (2 or 4)
    int kb_per_split;      // K blocks per split (multiple of nsub)
    int split;
    int nkb;               // total K blocks (K / 64)
    int col_tiles, batch_tiles, items;
    int issuers;           // MMA-issuing threads (1, 2 or 4)
    int bufs;              // accumulator sets (1 or 2)
    int a_slots;           // weight tiles in TMEM
    int code_slots;        // code ring depth (even)
    int x_slots;           // x ring depth (even)
    uint32_t code_slot_bytes, x_slot_bytes;
    uint32_t code_base;    // code ring offset (the x ring starts the shared memory)
    uint32_t scale_off, zero_off;  // offsets inside a code slot (codes at 0)
    int x3d;               // x of a stage is one 3-D box (else one 2-D box per block)
    int force_timeout;     // test hook: wait on a barrier nobody arrives at
    Epilogue epi;          // fused output epilogue (plain bf16 when mode == 0)
    const uint8_t* tag;    // the packed blob's tag
    uint32_t tag_want[4];
    size_t code_bytes;     // packed codes (bounds checks)
};

// ------------------------------------------------------------ kernel

struct SharedTail {
    uint64_t code_full[kMaxCodeSlots];      // codes, scales, zero-points of the stage landed
    uint64_t code_free[kMaxCodeSlots];      // read by the dequant warps (4 per block)
    uint64_t x_full[kMaxXSlots];            // x blocks of the stage landed
    uint64_t x_free[kMaxXSlots];            // MMAs of the stage finished (commit)
    uint64_t a_full[kMaxASlots];            // weight tile in TMEM (4 warp arrivals)
    uint64_t a_free[kMaxASlots];            // MMAs reading the weight tile finished (commit)
    uint64_t tmem_full[2];                  // accumulator set complete (one commit per issuer)
    uint64_t tmem_empty[2];                 // accumulator set drained (4 epilogue warps)
    uint64_t mma_done[kMaxIssuers];         // final drain of each issuer's MMAs
    uint64_t never;                         // test hook: nobody arrives here
    uint32_t tmem_base;
    int abort;
    int s_last;
};

struct Item {
    int col_tile, batch_tile, n0, b0, nvalid, kb_begin, nkb, ncs;
};

__device__ __forceinline__ Item decode_item(const Args& a, int it) {
    Item t;
    t.col_tile = it % a.col_tiles;
    const int rest = it / a.col_tiles;
    t.batch_tile = rest % a.batch_tiles;
    const int split_idx = rest / a.batch_tiles;
    t.n0 = t.col_tile * kTileN;
    t.b0 = t.batch_tile * a.bn;
    t.nvalid = min(kTileN, a.N - t.n0);
    t.kb_begin = split_idx * a.kb_per_split;
    t.nkb = min(a.kb_per_split, a.nkb - t.kb_begin);
    t.ncs = (t.nkb + a.nsub - 1) / a.nsub;
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

__device__ __forceinline__ int issuer_of_warp(int warp) {
    return (warp >= 1 && warp <= 3) ? warp - 1 : (warp == kIssuer3Warp ? 3 : -1);
}

// Weight copies of copy stage c of item t into a code slot: one bulk copy of
// the packed codes of its blocks (contiguous in the packed layout), one tensor
// copy of the scale rows of its groups and, for the asymmetric format, one of
// the zero-point rows.
template <bool kHasZeros>
__device__ __forceinline__ void issue_weight_copies(const Args& a, const CUtensorMap* smap,
                                                    const CUtensorMap* zmap, const Item& t,
                                                    int c, uint8_t* slot, uint32_t bar) {
    const int kb0 = t.kb_begin + c * a.nsub;
    const int ng = a.nsub > 1 ? a.nsub >> 1 : 1;
    uint32_t cb = (uint32_t)a.nsub * 2u * (uint32_t)t.nvalid * 16u;
    const size_t off = packed_tile_base(a.K, t.col_tile) + (size_t)(2 * kb0) * t.nvalid * 16;
    if (!in_bounds(off + cb <= a.code_bytes, a.status)) cb = 0;  // debug build: skip the copy
    const uint32_t zbytes = kHasZeros ? (uint32_t)ng * kZeroRowBytes : 0u;
    mbar_arrive_expect_tx(bar, cb + (uint32_t)ng * kScaleRowBytes + zbytes);
    if (cb != 0) bulk_g2s(smem_u32(slot), a.packed + off, cb, bar);
    tma_load_2d(smem_u32(slot + a.scale_off), smap, t.n0, kb0 >> 1, bar);
    if (kHasZeros) tma_load_2d(smem_u32(slot + a.zero_off), zmap, t.n0 >> 3, kb0 >> 1, bar);
}

// The x blocks of copy stage c into an x slot.
__device__ __forceinline__ void issue_x_copies(const Args& a, const CUtensorMap* xmap,
                                               const Item& t, int c, uint8_t* slot,
                                               uint32_t bar) {
    const int kb0 = t.kb_begin + c * a.nsub;
    mbar_arrive_expect_tx(bar, a.x_slot_bytes);
    if (a.x3d) {
        tma_load_3d(smem_u32(slot), xmap, 0, t.b0, kb0, bar);
    } else {
        for (int j = 0; j < a.nsub; ++j)
            tma_load_2d(smem_u32(slot + (size_t)j * a.bn * kBlockK * 2), xmap,
                        (kb0 + j) * kBlockK, t.b0, bar);
    }
}

template <bool kHasZeros, bool kFused, class Fmt>
__global__ void __launch_bounds__(kThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap smap,
          const __grid_constant__ CUtensorMap zmap, const Args a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled x tiles
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int RC = a.code_slots;
    const int RX = a.x_slots;
    const int SA = a.a_slots;
    const int I = a.issuers;
    SharedTail* tail = reinterpret_cast<SharedTail*>(smem + a.code_base +
                                                     (size_t)RC * a.code_slot_bytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = &tail->abort;
    auto x_slot = [&](int s) { return smem + (size_t)s * a.x_slot_bytes; };
    auto code_slot = [&](int s) { return smem + a.code_base + (size_t)s * a.code_slot_bytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < RC; ++s) {
            mbar_init(smem_u32(&tail->code_full[s]), 1);
            mbar_init(smem_u32(&tail->code_free[s]), 4 * a.nsub);
        }
        for (int s = 0; s < RX; ++s) {
            mbar_init(smem_u32(&tail->x_full[s]), 1);
            mbar_init(smem_u32(&tail->x_free[s]), a.nsub);  // one commit per block
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(smem_u32(&tail->a_full[s]), 4);
            mbar_init(smem_u32(&tail->a_free[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tail->tmem_full[b]), I);
            mbar_init(smem_u32(&tail->tmem_empty[b]), 4);
        }
        for (int i = 0; i < kMaxIssuers; ++i) mbar_init(smem_u32(&tail->mma_done[i]), 1);
        mbar_init(smem_u32(&tail->never), 1);
        tail->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&smap)) : "memory");
        if (kHasZeros)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&zmap))
                         : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tail->tmem_base)), "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tail->tmem_base;
    const uint32_t a_col0 = (uint32_t)(a.bufs * I * a.bn);  // weight tiles after the accumulators
    const uint32_t xblock_bytes = (uint32_t)a.bn * kBlockK * 2;
    // The next kernel on the stream may start now.  This one writes y and the
    // workspace, and reads x, only after the previous kernel has finished: the
    // producers wait before their first x copy, and everything else is ordered
    // after that through mbarriers.  The weights (codes, scales, zero-points)
    // do not depend on the previous kernel, so the first stages' weight copies
    // go out before.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int issuer = issuer_of_warp(warp);
    if (warp == 0 || warp == kProducer1Warp) {
        // ---------------- TMA producers: producer pr takes copy stages pr, pr+2, ...
        const int pr = warp == 0 ? 0 : 1;
        if (lane == 0 && pr == 0 && !blob_tag_matches(a.tag, a.tag_want))
            atomicExch(a.status, kStatusBadBlob);  // not a blob of this layout / shape
        if (lane == 0) {
            const Item first = decode_item(a, blockIdx.x);
            const int pre = min(RC, first.ncs);
            for (int c = pr; c < pre; c += 2)
                issue_weight_copies<kHasZeros>(a, &smap, &zmap, first, c, code_slot(c),
                                               smem_u32(&tail->code_full[c]));
            asm volatile("griddepcontrol.wait;" ::: "memory");
            int gcs = 0, done_c = 0, done_x = 0;  // stages walked; own stages issued (+1)
            Ring qc, qx;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x) {
                const Item t = decode_item(a, it);
                for (int c = 0; c < t.ncs; ++c, ++gcs, qc.next(RC), qx.next(RX)) {
                    if ((gcs & 1) != pr) continue;
                    if (gcs >= pre) {
                        // a code slot is free once the dequant warps read the stage RC back
                        if (gcs >= RC && !wait_fast(smem_u32(&tail->code_free[qc.s]), qc.ph ^ 1u,
                                                    abort, a.status)) {
                            ok = false;
                            break;
                        }
                        issue_weight_copies<kHasZeros>(a, &smap, &zmap, t, c, code_slot(qc.s),
                                                       smem_u32(&tail->code_full[qc.s]));
                        done_c = gcs + 1;
                    }
                    // an x slot is free once the MMAs of the stage RX back finished
                    if (gcs >= RX && !wait_fast(smem_u32(&tail->x_free[qx.s]), qx.ph ^ 1u, abort,
                                                a.status)) {
                        ok = false;
                        break;
                    }
                    issue_x_copies(a, &xmap, t, c, x_slot(qx.s), smem_u32(&tail->x_full[qx.s]));
                    done_x = gcs + 1;
                }
            }
            // After an expired wait, every copy in flight must land before the
            // CTA exits: wait for the latest use of every slot this producer filled.
            if (!ok) {
                const int last_c = max(done_c, pre);
                for (int c = max(0, last_c - RC); c < last_c; ++c)
                    if ((c & 1) == pr)
                        wait_bounded(smem_u32(&tail->code_full[c % RC]), (c / RC) & 1, abort,
                                     a.status, kTimeoutNs);
                for (int c = max(0, done_x - RX); c < done_x; ++c)
                    if ((c & 1) == pr)
                        wait_bounded(smem_u32(&tail->x_full[c % RX]), (c / RX) & 1, abort,
                                     a.status, kTimeoutNs);
            }
        }
    } else if (issuer >= 0) {
        // ---------------- MMA issuers: issuer i takes 64-row blocks i, i+I, ... (counted
        // over all items of the CTA; I divides the 4 dequant groups, so all blocks
        // of a group go to one issuer).  mbarrier waits test only the parity of a
        // phase, so every waiter must wait for a barrier's uses in order: each
        // dequant group has its own sub-ring of weight tiles, read by one issuer,
        // and every issuer reads every x slot it waits for in order (the x ring
        // depth times the blocks per stage is a multiple of I).
        if (lane == 0 && issuer < I) {
            const uint32_t idesc = instr_desc_f16kind(kTileN, a.bn, Fmt::kTcFormat);
            bool ok = true;
            if (a.force_timeout && issuer == 0)
                ok = wait_bounded(smem_u32(&tail->never), 0, abort, a.status,
                                  (unsigned long long)a.force_timeout * 1000000ull);
            // descriptor of x slot 0's first block; slot, block and K step add
            // to its start-address field (16-byte units, no carry out of it)
            const uint64_t desc0 = smem_desc_sw128(smem_u32(smem));
            const uint32_t slot16 = a.x_slot_bytes >> 4;
            const uint32_t xblock16 = xblock_bytes >> 4;
            const int SAg = SA >> 2;  // tiles per dequant group
            // block 4k + g is group g's k-th block: all groups' sub-rings are at the
            // same position, stepped once every 4 blocks
            Ring qx, qk;
            int buf = 0, use = 0;
            int gb = 0;  // blocks walked
            for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x) {
                const Item t = decode_item(a, it);
                if (use >= 1 && !wait_bounded(smem_u32(&tail->tmem_empty[buf]), (use - 1) & 1,
                                              abort, a.status, kTimeoutNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tmem_d = tmem_base + (uint32_t)((buf * I + issuer) * a.bn);
                bool first = true;
                for (int c = 0; ok && c < t.ncs; ++c, qx.next(RX)) {
                    const uint64_t sdesc = desc0 + (uint64_t)((uint32_t)qx.s * slot16);
                    for (int j = 0; j < a.nsub; ++j, ++gb) {
                        const int g = gb & (kDequantGroups - 1);
                        const int sa = g * SAg + qk.s;
                        const uint32_t pha = qk.ph;
                        if (g == kDequantGroups - 1) qk.next(SAg);
                        if ((gb & (I - 1)) != issuer) continue;
                        if (!wait_fast(smem_u32(&tail->x_full[qx.s]), qx.ph, abort, a.status) ||
                            !wait_fast(smem_u32(&tail->a_full[sa]), pha, abort, a.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t tmem_a = tmem_base + a_col0 + (uint32_t)(sa * kACols);
                        const uint64_t bdesc = sdesc + (uint64_t)((uint32_t)j * xblock16);
#pragma unroll
                        for (int kk = 0; kk < kBlockK / 16; ++kk)
                            mma_bf16_ts(tmem_d, tmem_a + 8 * kk, bdesc + (uint64_t)(2 * kk),
                                        idesc, (first && kk == 0) ? 0u : 1u);
                        first = false;
                        mma_commit(smem_u32(&tail->a_free[sa]));
                        mma_commit(smem_u32(&tail->x_free[qx.s]));  // one of nsub per stage
                    }
                }
                if (!ok) break;
                mma_commit(smem_u32(&tail->tmem_full[buf]));  // fires once these MMAs are done
                if (++buf == a.bufs) {
                    buf = 0;
                    ++use;
                }
            }
            if (!ok) {
                // let the epilogue drain: the accumulator sets "complete" once
                // every issued MMA has finished
                mma_commit(smem_u32(&tail->tmem_full[0]));
                mma_commit(smem_u32(&tail->tmem_full[1]));
            }
            // every MMA of this thread has finished before TMEM is released, also
            // after an abort (issued MMAs wait on nothing, so this wait is short)
            mma_commit(smem_u32(&tail->mma_done[issuer]));
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(&tail->mma_done[issuer]), 0) &&
                   globaltimer() - t0 < kTimeoutNs) {
            }
        }
    } else if (warp >= kDequantWarp0) {
        // ---------------- dequant: group grp takes blocks grp, grp+4, ... into its own
        // sub-ring of weight tiles; each thread owns one weight column of the
        // tile = one TMEM lane.  Waits on a code slot stay in order: with
        // nsub = 4 every group reads every stage, with nsub = 2 a pair of groups
        // reads every other stage and the code ring depth is even.
        const int dw = warp - kDequantWarp0;
        const int grp = dw >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16) + a_col0;
        int g4 = 0;  // blocks walked, modulo the group count
        const int SAg = SA >> 2;
        Ring q, qa;  // code ring; this group's sub-ring of weight tiles
        int own = 0;  // blocks of this group so far
        bool ok = true;
        for (int it = blockIdx.x; ok && it < a.items; it += gridDim.x) {
            const Item t = decode_item(a, it);
            const int rr = min(r, t.nvalid - 1);  // lanes past a ragged edge repeat a column
            for (int c = 0; ok && c < t.ncs; ++c, q.next(RC)) {
                const int nblk = a.nsub;
                for (int j = 0; j < nblk; ++j) {
                    const bool mine = g4 == grp;
                    if (++g4 == kDequantGroups) g4 = 0;
                    if (!mine) continue;
                    const int sa = grp * SAg + qa.s;
                    bool landed = wait_fast(smem_u32(&tail->code_full[q.s]), q.ph, abort, a.status);
                    // the tile slot is free once this group's block SA/4 back finished
                    if (landed && own >= SAg)
                        landed = wait_fast(smem_u32(&tail->a_free[sa]), qa.ph ^ 1u, abort,
                                           a.status);
                    if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform exit
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* slot = code_slot(q.s);
                    const uint4* codes = reinterpret_cast<const uint4*>(slot) +
                                         (size_t)(2 * j) * t.nvalid;
                    // chunks 2(kb0 + j) and 2(kb0 + j) + 1 (swizzled runs)
                    const int swz = packed_swizzle(2 * (t.kb_begin + c * a.nsub + j));
                    const uint4 q0 = codes[rr ^ swz];
                    const uint4 q1 = codes[t.nvalid + (rr ^ (swz + 2))];
                    const int kb0 = t.kb_begin + c * a.nsub;
                    const int grow = ((kb0 + j) >> 1) - (kb0 >> 1);  // group row inside the stage
                    const uint32_t s2 = scale_pair(reinterpret_cast<const uint16_t*>(
                        slot + a.scale_off + grow * kScaleRowBytes)[rr]);
                    uint32_t z2 = Fmt::kSymZero2;
                    if (kHasZeros) {
                        const uint32_t zw = reinterpret_cast<const uint32_t*>(
                            slot + a.zero_off + grow * kZeroRowBytes)[rr >> 3];
                        z2 = zero_pair<Fmt>((zw >> (4 * (rr & 7))) & 0xFu);
                    }
                    // chunk h (rows 32h .. 32h+31 of the block) -> TMEM columns 16h .. 16h+15
                    const uint32_t col = lane_addr + (uint32_t)(sa * kACols);
                    {
                        const uint32_t words[4] = {q0.x, q0.y, q0.z, q0.w};
                        uint32_t v[16];
#pragma unroll
                        for (int jw = 0; jw < 4; ++jw)
#pragma unroll
                            for (int pp = 0; pp < 4; ++pp)
                                v[4 * jw + pp] = dequant_pair<Fmt>(words[jw], pp, z2, s2);
                        tmem_st_16(col, v);
                    }
                    {
                        const uint32_t words[4] = {q1.x, q1.y, q1.z, q1.w};
                        uint32_t v[16];
#pragma unroll
                        for (int jw = 0; jw < 4; ++jw)
#pragma unroll
                            for (int pp = 0; pp < 4; ++pp)
                                v[4 * jw + pp] = dequant_pair<Fmt>(words[jw], pp, z2, s2);
                        tmem_st_16(col + 16, v);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&tail->a_full[sa]));
                        mbar_arrive(smem_u32(&tail->code_free[q.s]));  // codes read
                    }
                    qa.next(SAg);
                    ++own;
                }
            }
        }
    } else if (warp >= kEpilogueWarp0) {
        // ---------------- epilogue (TMEM lane quadrant = warp % 4)
        const int quad = warp & 3;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
        int j = 0;
        int g0 = 0;  // first block of the item (counted over the CTA's items) modulo I
        for (int it = blockIdx.x; it < a.items; it += gridDim.x, ++j) {
            const Item t = decode_item(a, it);
            const int buf = a.bufs == 2 ? (j & 1) : 0;
            const int use = a.bufs == 2 ? (j >> 1) : j;
            const bool done = wait_bounded(smem_u32(&tail->tmem_full[buf]), use & 1, abort,
                                           a.status, kTimeoutNs);
            tc_fence_after();
            const bool live = __all_sync(0xffffffffu, done && !*abort);
            if (live) {  // tcgen05.ld is warp-collective
                const int nn = t.n0 + quad * 32 + lane;
                // issuer i received blocks of this item iff (i - g0) mod I < nkb;
                // the item's first block went to issuer g0
                const uint32_t acc0 = lane_base + (uint32_t)(buf * I * a.bn);
                for (int c0 = 0; c0 < a.bn; c0 += 16) {
                    float v[16];
                    uint32_t r[16];
                    tmem_ld_16_async(acc0 + (uint32_t)(g0 * a.bn) + c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) v[jj] = __uint_as_float(r[jj]);
                    for (int k = 1; k < min(I, t.nkb); ++k) {
                        const int i = g0 + k < I ? g0 + k : g0 + k - I;
                        tmem_ld_16_async(acc0 + (uint32_t)(i * a.bn) + c0, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) v[jj] += __uint_as_float(r[jj]);
                    }
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
                                    a.y[(size_t)b * a.N + nn] = (uint16_t)Fmt::from_f32(v[jj]);
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
            if (lane == 0) mbar_arrive(smem_u32(&tail->tmem_empty[buf]));
            if (!live) break;
            g0 = (g0 + t.nkb) % I;
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
                    // 4 columns per thread and 4 loads in flight: the sums come
                    // back from L2, so latency, not bandwidth, sets the pace
                    const int rows = min(a.bn, a.B - t.b0);
                    const int c4n = t.nvalid / 4;
                    const int total = rows * c4n;
                    const int et = threadIdx.x - 32 * kEpilogueWarp0;
                    for (int e0 = et; e0 < total; e0 += 128 * 4) {
                        float4 v[4];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int e = e0 + 128 * jj;
                            if (e < total) {
                                const int rr = e / c4n, cc = 4 * (e - (e / c4n) * c4n);
                                if (in_bounds(t.b0 + rr < a.B && t.n0 + cc + 4 <= a.N, a.status))
                                    v[jj] = __ldcg(reinterpret_cast<const float4*>(
                                        a.partial + (size_t)(t.b0 + rr) * a.N + t.n0 + cc));
                            }
                        }
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int e = e0 + 128 * jj;
                            if (e < total) {
                                const int rr = e / c4n, cc = 4 * (e - (e / c4n) * c4n);
                                const size_t off = (size_t)(t.b0 + rr) * a.N + t.n0 + cc;
                                if (t.b0 + rr >= a.B || t.n0 + cc + 4 > a.N) continue;
                                if constexpr (kFused)
                                    epi_store4_fused(a.y, a.N, t.b0 + rr, t.n0 + cc, v[jj].x, v[jj].y,
                                           v[jj].z, v[jj].w, a.epi);
                                else
                                    epi_store4_plain<Fmt>(a.y, a.N, t.b0 + rr, t.n0 + cc, v[jj].x, v[jj].y,
                                           v[jj].z, v[jj].w, a.epi);
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

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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

// Shared memory: [x ring: x_slots x (nsub x tiles of bn x 128 B)]
// [code ring: code_slots x (codes nsub x 4 KB, scale rows, zero-point rows)][tail].
// Both ring depths are even: consecutive uses of a slot fall to the same
// producer, and (nsub = 2) to the same pair of dequant groups, so every
// waiter's waits on a slot stay in order.
struct RingLayout {
    uint32_t x_slot_bytes, code_slot_bytes, scale_off, zero_off, code_base;
    int x_slots, code_slots;
    size_t smem;
};

RingLayout ring_layout(int bn, int nsub) {
    RingLayout l;
    const int ng = nsub > 1 ? nsub / 2 : 1;
    l.x_slot_bytes = (uint32_t)nsub * (uint32_t)bn * kBlockK * 2;  // multiple of 1024
    l.scale_off = (uint32_t)nsub * kCodeBlockBytes;
    l.zero_off = l.scale_off + (uint32_t)ng * kScaleRowBytes;
    l.code_slot_bytes = (l.zero_off + (uint32_t)ng * kZeroRowBytes + 127u) & ~127u;
    const size_t avail = kSmemBudget - 1024 - sizeof(SharedTail);
    // the deepest balanced pair of rings (then the most slots) that fits
    int best_c = 0, best_x = 0;
    for (int c = 2; c <= kMaxCodeSlots; c += 2) {
        if ((size_t)c * l.code_slot_bytes > avail) break;
        int x = (int)std::min<size_t>(kMaxXSlots, (avail - (size_t)c * l.code_slot_bytes) /
                                                      l.x_slot_bytes) & ~1;
        if (x < 2) continue;
        const int m = std::min(c, x), bm = std::min(best_c, best_x);
        if (m > bm || (m == bm && c + x > best_c + best_x)) {
            best_c = c;
            best_x = x;
        }
    }
    l.code_slots = best_c;
    l.x_slots = best_x;
    l.code_base = (uint32_t)best_x * l.x_slot_bytes;
    l.smem = (size_t)l.code_base + (size_t)best_c * l.code_slot_bytes + sizeof(SharedTail) + 1024;
    return l;
}

}  // namespace

bool tc_available() {
    // cached per device: sm_103 and the tensor-map encoder are both needed
    static std::mutex mu;
    static int known[64] = {0};  // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (known[dev] == 0) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        known[dev] = (major == 10 && minor == 3 && encode_fn() != nullptr) ? 1 : 2;
    }
    return known[dev] == 1;
}

TcPlan plan_tc(int B, int K, int N, int num_sms) {
    if (B > kMaxTmemBatch) {
        TcPlan w = plan_tc_wide(B, K, N, num_sms);
        w.wide = true;
        return w;
    }
    TcPlan p{};
    p.batch_tiles = (B + 255) / 256;
    const int per = (B + p.batch_tiles - 1) / p.batch_tiles;
    p.bn = std::min(256, (per + 15) / 16 * 16);
    // MMAs of one thread run in order and a short MMA (small bn) costs about as
    // long as a long one, so small tiles spread their copy stages over several
    // issuers; TMEM (512 columns) holds bufs x issuers accumulators of bn
    // columns plus the ring of weight tiles (32 columns each).
    if (p.bn <= 32) {
        p.issuers = 4;
        p.bufs = 2;
    } else if (p.bn <= 64) {
        p.issuers = 4;
        p.bufs = 1;
    } else if (p.bn <= 128) {
        p.issuers = 2;
        p.bufs = 1;
    } else {
        p.issuers = 1;
        p.bufs = 1;
    }
    // a multiple of the dequant group count, so a tile slot's consecutive uses
    // fall to the same group (its waits on the slot stay in order)
    p.a_slots = std::min(kMaxASlots, (kTmemCols - p.bufs * p.issuers * p.bn) / kACols) / 4 * 4;
    // copy stages of 256 K rows (16 KB of codes) while the x blocks are small,
    // else 128 rows; every stage is whole (nsub divides the K blocks)
    p.col_tiles = (N + kTileN - 1) / kTileN;
    const int nkb = K / kBlockK;
    p.nsub = (p.bn <= 32 && nkb % 4 == 0) ? 4 : 2;
    const long long tiles = (long long)p.col_tiles * p.batch_tiles;
    // persistent CTAs (one per SM) take items round robin; choose the K split
    // (whole copy stages per split) minimising the busiest CTA's K blocks plus
    // a fixed cost per item and a small cost per split (accumulator traffic)
    double best = 1e300;
    int best_split = 1, best_kbps = (nkb + p.nsub - 1) / p.nsub * p.nsub;
    for (int split = 1; split <= std::min(16, nkb); ++split) {
        const int kbps = ((nkb + split - 1) / split + p.nsub - 1) / p.nsub * p.nsub;
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

size_t tc_workspace_bytes(const TcPlan& p, int B, int N) {
    return p.split > 1 ? kCounterBytes + (size_t)B * N * sizeof(float) : 0;
}

static cudaError_t launch_tc_impl(const TcPlan& p, const void* x, const void* packed,
                                  const void* scales, bool has_zeros, void* y, int B, int K,
                                  int N, void* workspace, unsigned int* status,
                                  int force_timeout_ms, const Epilogue& epi,
                                  cudaStream_t stream) {
    if (p.wide) {
        // The wide kernel serves more than 16 batch rows, whose tiles its
        // planner makes at least 32 rows tall; 16-row tiles are refused: a
        // timing-only build that ran them (4096 -> 128256 at 8 rows) reported
        // a device error, most likely from a y tensor store whose box was
        // taller than the whole output.
        if (p.bn < 32) return cudaErrorInvalidConfiguration;
        return launch_tc_wide(p, x, packed, scales, has_zeros, y, B, K, N, workspace, status,
                              force_timeout_ms, epi, stream);
    }
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const int ng = p.nsub > 1 ? p.nsub / 2 : 1;
    const cuuint32_t e1[3] = {1, 1, 1};
    // x: 3-D view (k within a block, row, block) so one box brings a stage's
    // nsub blocks, each a 1024-byte-aligned bn x 128-byte swizzled tile; if the
    // encoder refuses the view, one 2-D box per block
    CUtensorMap xmap;
    int x3d = 1;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)kBlockK, (cuuint64_t)B, (cuuint64_t)(K / kBlockK)};
        const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)kBlockK * 2};
        const cuuint32_t box[3] = {(cuuint32_t)kBlockK, (cuuint32_t)p.bn, (cuuint32_t)p.nsub};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides,
                box, e1, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            x3d = 0;
            const cuuint64_t dims2[2] = {(cuuint64_t)K, (cuuint64_t)B};
            const cuuint64_t strides2[1] = {(cuuint64_t)K * 2};
            const cuuint32_t box2[2] = {(cuuint32_t)kBlockK, (cuuint32_t)p.bn};
            if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims2,
                    strides2, box2, e1, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
    }
    // scales [K/128][N] (bf16, or fp16: the copies move 16-bit patterns, so one
    // map type serves both formats): box of 128 columns x ng group rows
    CUtensorMap smap;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)(K / kGroup)};
        const cuuint64_t strides[1] = {(cuuint64_t)N * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kTileN, (cuuint32_t)ng};
        if (enc(&smap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(scales), dims,
                strides, box, e1, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // zero-points: padded uint32 rows after the codes; box of 16 words x ng rows
    CUtensorMap zmap = smap;
    if (has_zeros) {
        const int row_words = packed_zero_row_words(N);
        const cuuint64_t dims[2] = {(cuuint64_t)row_words, (cuuint64_t)(K / kGroup)};
        const cuuint64_t strides[1] = {(cuuint64_t)row_words * 4};
        const cuuint32_t box[2] = {(cuuint32_t)(kTileN / 8), (cuuint32_t)ng};
        void* zbase = static_cast<char*>(const_cast<void*>(packed)) + packed_code_bytes(K, N);
        if (enc(&zmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, zbase, dims, strides, box, e1,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    const RingLayout lay = ring_layout(p.bn, p.nsub);
    Args a;
    a.packed = static_cast<const uint8_t*>(packed);
    a.y = static_cast<uint16_t*>(y);
    a.partial = ws_partials(workspace);
    a.counters = ws_counters(workspace);
    a.status = status;
    a.B = B;
    a.K = K;
    a.N = N;
    a.bn = p.bn;
    a.nsub = p.nsub;
    a.kb_per_split = p.kb_per_split;
    a.split = p.split;
    a.nkb = K / kBlockK;
    a.col_tiles = p.col_tiles;
    a.batch_tiles = p.batch_tiles;
    a.items = p.col_tiles * p.batch_tiles * p.split;
    a.issuers = p.issuers;
    a.bufs = p.bufs;
    a.a_slots = p.a_slots;
    a.code_slots = lay.code_slots;
    a.x_slots = lay.x_slots;
    a.code_slot_bytes = lay.code_slot_bytes;
    a.x_slot_bytes = lay.x_slot_bytes;
    a.code_base = lay.code_base;
    a.scale_off = lay.scale_off;
    a.zero_off = lay.zero_off;
    a.x3d = x3d;
    a.force_timeout = force_timeout_ms;
    a.epi = epi;
    a.tag = a.packed + packed_tag_offset(K, N, has_zeros);
    a.code_bytes = code_bound_bytes(K, N);
    {
        const BlobTag want = blob_tag(K, N, has_zeros);
        for (int i = 0; i < 4; ++i) a.tag_want[i] = want.w[i];
    }
    if (a.a_slots < 4 || a.code_slots < 2 || a.x_slots < 2) return cudaErrorInvalidConfiguration;

    const size_t smem = lay.smem;
    const bool fused = epi.mode != 0;
    const void* kern =
        epi.f16 ? (has_zeros ? reinterpret_cast<const void*>(tc_kernel<true, false, F16>)
                             : reinterpret_cast<const void*>(tc_kernel<false, false, F16>))
        : has_zeros ? (fused ? reinterpret_cast<const void*>(tc_kernel<true, true, Bf16>)
                             : reinterpret_cast<const void*>(tc_kernel<true, false, Bf16>))
                    : (fused ? reinterpret_cast<const void*>(tc_kernel<false, true, Bf16>)
                             : reinterpret_cast<const void*>(tc_kernel<false, false, Bf16>));
    cudaError_t err =
        set_smem_limit(kern, smem);
    if (err != cudaSuccess) return err;
    void* args[] = {&xmap, &smap, &zmap, &a};
    const int grid = std::min(a.items, p.grid);
    return launch_with_pdl(kern, dim3(grid), dim3(kThreads), smem, stream, args);
}

cudaError_t launch_tc(const TcPlan& p, const void* x, const void* packed, const void* scales,
                      bool has_zeros, void* y, int B, int K, int N, void* workspace,
                      unsigned int* status, const Epilogue& epi, cudaStream_t stream) {
    return launch_tc_impl(p, x, packed, scales, has_zeros, y, B, K, N, workspace, status, 0,
                          epi, stream);
}

cudaError_t launch_tc_forced_timeout(const TcPlan& p, const void* x, const void* packed,
                                     const void* scales, bool has_zeros, void* y, int B, int K,
                                     int N, void* workspace, unsigned int* status, int wait_ms,
                                     cudaStream_t stream) {
    return launch_tc_impl(p, x, packed, scales, has_zeros, y, B, K, N, workspace, status,
                          wait_ms, Epilogue{}, stream);
}

}  // namespace w4a16
