// skinny.cu -- memory-bound small-batch W4A16 GEMM (decode, B <= 32).
//
// At small B the layer is a weight stream: every weight is read once from HBM
// and used B times ("When quantization pays -- and when it does not", model of
// a decode step: the memory term W*b_w/beta dominates until the batch reaches
// the ridge).  At GB300's memory latency, HBM speed needs on the order of
// 100 KB of loads in flight per SM -- far more than registers can hold -- so
// the weights stream through shared memory:
//
//  * persistent CTAs, one producer warp + 8 consumer warps.  The producer's
//    lane 0 bulk-copies (cp.async.bulk) one contiguous 16 KB block of packed
//    codes per ring slot (two 128-row groups of a 128-column tile); its 32
//    lanes copy the matching activations, scales and zero-points with
//    cp.async and attach them to the slot's mbarrier (arrive.noinc);
//  * each consumer warp owns 16 columns of the tile: it reads its codes from
//    the slot (one conflict-free 16-byte load per lane per chunk), turns them
//    into the exact integers (q - z) with the shared magic-number OR and an
//    exact bf16 subtraction, and feeds those as the A operand of warp-level
//    m16n8k16 tensor-core products in which the 16 rows are weight columns
//    and the 8 columns batch rows (operands swapped, so the batch pads only to
//    8).  The products (q - z)*x are exact; each 128-row group is summed in
//    fp32 and multiplied by its scale once (acc += s * sum), which removes the
//    per-weight bf16 multiply from the CUDA cores -- at decode batch sizes the
//    decode instructions and their latency, not the tensor cores, bound the
//    kernel.  The k order inside an mma is
//    free, so each lane's four k values per step are consecutive rows of its
//    own 32-row chunk; the activations are staged in exactly that fragment
//    order, which makes each fragment load one 16-byte read;
//  * work units are (batch chunk, column tile, K split), handed out
//    dynamically (the first unit of each CTA is fixed, later ones come from an
//    atomic work counter), so slow and fast SMs even out; the producer decodes
//    a unit once and publishes, per slot, what the consumers need;
//  * grouped mode (mixture-of-experts layers): the batch chunks are counted
//    over all experts from a device-side routing table, and a unit's codes,
//    scales and rows are its expert's;
//  * a dedicated epilogue warp takes each finished unit's accumulators from
//    shared memory and writes y -- or, for a K split, adds them into an fp32
//    accumulator with vector reductions (red.global.add.v4.f32), the last
//    unit of a tile to arrive (arrival counter) converting the sum to bf16
//    and clearing the accumulator; the order of the fp32 additions across
//    K splits follows arrival order -- while the consumers already work on
//    the next unit;
//  * programmatic dependent launch: the first ring slots' weight copies are
//    issued before waiting for the previous kernel on the stream, so
//    consecutive layers' weight streams overlap.
// The plain, grouped and fused-epilogue (bias / SiLU gate) forms are separate
// instantiations, so the plain kernel carries none of the others' code.
// Every mbarrier wait is bounded; on expiry the kernel records
// W4A16_ERR_TIMEOUT in the device status word and returns.
#include <cuda_runtime.h>

#include <algorithm>

#include "checks.cuh"
#include "dequant.cuh"
#include "epilogue.cuh"
#include "launch.cuh"

namespace w4a16 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (2 + kConsumerWarps);  // 320
constexpr int kTileCols = kPackTileCols;             // 128 columns per tile
constexpr int kSlotGroups = 2;                       // 128-row groups per ring slot
constexpr uint32_t kSlotCodeBytes = kSlotGroups * 4 * kTileCols * 16;  // 16 KB
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr unsigned int kStatusTimeout = 7;           // W4A16_ERR_TIMEOUT
constexpr int kWorkCounter = kMaxCounters - 2;       // workspace words used by the scheduler
constexpr int kDoneCounter = kMaxCounters - 1;

// Up to 8 rows: three CTAs per SM (3 slots each, 64 registers, no spills)
// hide more of the consumers' latency than two CTAs with 4 slots (measured:
// decode-layer step 312 -> 301 us); 16 rows: two CTAs; 32 rows: one.
template <int NT> constexpr int ring_slots() { return NT == 1 ? 3 : (NT == 2 ? 3 : 5); }
template <int NT> constexpr int ctas_per_sm_t() { return NT >= 4 ? 1 : (NT == 1 ? 3 : 2); }
template <int NT> constexpr uint32_t slot_x_bytes() { return kSlotGroups * 16 * 8 * NT * 16; }
constexpr uint32_t kSlotScaleBytes = kSlotGroups * kTileCols * 2;  // 512
constexpr uint32_t kSlotZeroBytes = kSlotGroups * kTileCols / 2;   // 128
template <int NT> constexpr uint32_t slot_bytes() {
    return kSlotCodeBytes + slot_x_bytes<NT>() + kSlotScaleBytes + kSlotZeroBytes;
}
// accumulators of one unit: [warp][bt][i][lane]
template <int NT> constexpr uint32_t result_bytes() { return kConsumerWarps * NT * 4 * 32 * 4; }

struct Args {
    const uint16_t* x;
    const uint8_t* packed;
    const uint16_t* scales;
    const uint32_t* zeros;
    uint16_t* y;
    float* partial;      // fp32 accumulator [B][N], zero between calls (split > 1)
    uint32_t* counters;  // fixed workspace prefix: per-tile arrivals + scheduler words
    unsigned int* status;
    int B, K, N;
    int tiles, split, gps, units;
    // grouped (mixture-of-experts) GEMM: offsets != nullptr.  Rows
    // offsets[e] .. offsets[e+1]-1 of x and y belong to expert e, whose packed
    // blob and scales sit w_stride bytes / s_stride scales after expert e-1's;
    // B is the total row count, units is then counted on the device.
    const int* offsets;
    int E;
    size_t w_stride, s_stride;
    Epilogue epi;        // fused output epilogue (plain bf16 when mode == 0)
    const uint8_t* tag;  // the packed blob's tag (the first expert's when grouped)
    uint32_t tag_want[4];
    size_t code_bytes;   // packed codes of one expert (bounds checks)
    int zrow_words;      // words per padded zero-point row (bounds checks)
};

constexpr int kMaxExperts = 256;

struct Tail {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t res_full[2];
    uint64_t res_empty[2];
    int slot_unit[8];    // unit of each ring slot (-1: no more work)
    int slot_step[8];    // step of the unit held by the slot
    int slot_meta[8];    // what the consumers need of it (slot_meta_pack)
    int res_unit[2];
    int abort;
    int total_units;                     // units of this call
    // grouped: expert e owns rows row_start[e] .. row_start[e+1]-1 and the
    // batch chunks chunk_prefix[e] .. chunk_prefix[e+1]-1
    int row_start[kMaxExperts + 1];
    int chunk_prefix[kMaxExperts + 1];
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait; false when this CTA is aborting or the wait expired (then it
// sets the abort flag and the device status word).
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status) {
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > kTimeoutNs) {
            *abort = 1;
            atomicExch(status, kStatusTimeout);
            return false;
        }
    }
}

// warp-uniform bounded wait
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status) {
    return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort, status));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Warp-level m16n8k16 product with fp32 accumulation, bf16 or fp16 operands.
template <class Fmt>
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (Fmt::kIsF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Work unit u -> (batch chunk, tile, split index) and its extents.  bc counts
// batch chunks over all experts (it indexes the split-K arrival counters);
// b0 is the unit's first row of x and y; packed / scales / zeros point at the
// unit's expert.
struct Unit {
    int bc, tile, sk, g_begin, ng, n0, width, b0, rows, nsteps;
    const uint8_t* packed;
    const uint16_t* scales;
    const uint32_t* zeros;
};

// Four fp32 values -> four 16-bit values (RNE) at a 8-byte aligned address.
template <class Fmt>
__device__ __forceinline__ void store4(uint16_t* dst, float v0, float v1, float v2, float v3) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(Fmt::from_f32(v0) | (Fmt::from_f32(v1) << 16),
                                                Fmt::from_f32(v2) | (Fmt::from_f32(v3) << 16));
}

// A slot's unit as the consumers see it, decoded once by the producer (the
// unit decode's integer divisions would otherwise run in every consumer warp
// at every step): tile width, groups in the slot, batch rows, last step.
__device__ __forceinline__ int slot_meta_pack(int width, int ngs, int rows, bool last) {
    return width | (ngs << 8) | (rows << 12) | ((last ? 1 : 0) << 20);
}

// Kernel variants (compiled separately so the plain kernel carries no code
// of the others): plain, grouped (mixture of experts), fused epilogue.
constexpr int kPlain = 0, kGrouped = 1, kFusedEpi = 2;

template <int NT, int kMode>
__device__ __forceinline__ Unit decode_unit(const Args& a, const Tail* t, int u) {
    constexpr int kRows = 8 * NT;
    Unit w;
    w.sk = u % a.split;
    const int rest = u / a.split;
    w.tile = rest % a.tiles;
    w.bc = rest / a.tiles;
    w.g_begin = w.sk * a.gps;
    w.ng = min(a.gps, a.K / kGroup - w.g_begin);
    w.n0 = w.tile * kTileCols;
    w.width = packed_tile_width(a.N, w.tile);
    w.nsteps = (w.ng + kSlotGroups - 1) / kSlotGroups;
    if constexpr (kMode != kGrouped) {
        w.b0 = w.bc * kRows;
        w.rows = min(kRows, a.B - w.b0);
        w.packed = a.packed;
        w.scales = a.scales;
        w.zeros = a.zeros;
    } else {
        // the expert whose chunks hold bc (chunk_prefix is non-decreasing)
        int lo = 0, hi = a.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (t->chunk_prefix[mid] <= w.bc) lo = mid;
            else hi = mid - 1;
        }
        const int e = lo;
        w.b0 = t->row_start[e] + (w.bc - t->chunk_prefix[e]) * kRows;
        w.rows = min(kRows, t->row_start[e + 1] - w.b0);
        w.packed = a.packed + (size_t)e * a.w_stride;
        w.scales = a.scales + (size_t)e * a.s_stride;
        w.zeros = reinterpret_cast<const uint32_t*>(w.packed + ((const uint8_t*)a.zeros - a.packed));
    }
    return w;
}

// ------------------------------------------------------------ kernel

template <int NT, bool kHasZeros, int kMode, class Fmt>
__global__ void __launch_bounds__(kThreads, ctas_per_sm_t<NT>())
skinny_kernel(const Args a) {
    constexpr int kRows = 8 * NT;
    constexpr int S = ring_slots<NT>();
    extern __shared__ __align__(128) uint8_t smem[];
    float* res = reinterpret_cast<float*>(smem + S * slot_bytes<NT>());
    Tail* tail = reinterpret_cast<Tail*>(smem + S * slot_bytes<NT>() + 2 * result_bytes<NT>());
    volatile int* abort = &tail->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto slot_codes = [&](int s) { return smem + s * slot_bytes<NT>(); };
    auto slot_x = [&](int s) {
        return reinterpret_cast<uint4*>(smem + s * slot_bytes<NT>() + kSlotCodeBytes);
    };
    auto slot_scales = [&](int s) {
        return reinterpret_cast<uint16_t*>(smem + s * slot_bytes<NT>() + kSlotCodeBytes +
                                           slot_x_bytes<NT>());
    };
    auto slot_zeros = [&](int s) {
        return reinterpret_cast<uint32_t*>(smem + s * slot_bytes<NT>() + kSlotCodeBytes +
                                           slot_x_bytes<NT>() + kSlotScaleBytes);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // lane 0's arrive (with the expected bytes) + one cp.async arrive per producer lane
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&tail->full[s])),
                         "r"(33));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&tail->empty[s])),
                         "r"(kConsumerWarps));
        }
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                         ::"r"(smem_u32(&tail->res_full[b])), "r"(kConsumerWarps));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                         ::"r"(smem_u32(&tail->res_empty[b])), "r"(1));
        }
        tail->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (kMode == kGrouped) {
        // grouped: the routing table may be written by the previous kernel on
        // the stream, so wait for it before the first read
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (warp == 0) {
            // Row boundaries m_i = max(clamp(offsets[j], 0, B), j <= i): the
            // experts' row ranges are then disjoint and inside x and y whatever
            // the table holds, and there are at most min(B, B/kRows + E) batch
            // chunks (the counter prefix is sized for that).  Lane l owns
            // boundaries 8l+1 .. 8l+8; two warp scans (max, then sum).
            constexpr int kPer = kMaxExperts / 32;
            const int b_first = min(max(__ldg(a.offsets), 0), a.B);
            int m[kPer];
            int run = 0;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int i = kPer * lane + j + 1;
                const int v = i <= a.E ? min(max(__ldg(a.offsets + i), 0), a.B) : 0;
                run = max(run, v);
                m[j] = run;
            }
            int incl = run;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl = max(incl, o);
            }
            int before = __shfl_up_sync(0xffffffffu, incl, 1);
            before = lane == 0 ? b_first : max(before, b_first);
            int chunks[kPer];
            int csum = 0;
            int prev = before;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                m[j] = max(m[j], before);
                chunks[j] = (kPer * lane + j < a.E) ? (m[j] - prev + kRows - 1) / kRows : 0;
                csum += chunks[j];
                prev = m[j];
            }
            int cincl = csum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, cincl, d);
                if (lane >= d) cincl += o;
            }
            int c = cincl - csum;
            if (lane == 0) {
                tail->row_start[0] = b_first;
                tail->chunk_prefix[0] = 0;
            }
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int i = kPer * lane + j + 1;
                c += chunks[j];
                if (i <= a.E) {
                    tail->row_start[i] = m[j];
                    tail->chunk_prefix[i] = c;
                }
            }
            if (lane == 31) tail->total_units = cincl * a.tiles * a.split;
        }
    } else if (threadIdx.x == 0) {
        tail->total_units = a.units;
    }
    __syncthreads();
    const int total_units = tail->total_units;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ---------------- producer
        uint64_t evict_first;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
        int step = 0;        // ring position
        int issued = 0;      // ring positions fully issued
        int w_issued = 0;    // ring positions whose code copy is issued
        bool ok = true;
        if (lane == 0 && !blob_tag_matches(a.tag, a.tag_want))
            atomicExch(a.status, kStatusBadBlob);  // not a blob of this layout / shape
        // The first unit is fixed (blockIdx.x): its first slots' code copies go
        // out before waiting for the previous kernel on the stream.
        const bool has_first = (int)blockIdx.x < total_units;
        const Unit first = decode_unit<NT, kMode>(a, tail, has_first ? (int)blockIdx.x : 0);
        const uint8_t* first_codes = first.packed + packed_tile_base(a.K, first.tile);
        auto issue_codes = [&](const Unit& w, const uint8_t* tile_codes, int st, int pos) {
            const int s = pos % S;
            const int g0 = w.g_begin + st * kSlotGroups;
            const int ngs = min(kSlotGroups, w.g_begin + w.ng - g0);
            uint32_t bytes = (uint32_t)ngs * 4 * w.width * 16;
            const uint8_t* src = tile_codes + (size_t)(4 * g0) * w.width * 16;
            if (!in_bounds(src >= w.packed && src + bytes <= w.packed + a.code_bytes, a.status))
                bytes = 0;  // debug build: skip the copy (the barrier still completes)
            const uint32_t full = smem_u32(&tail->full[s]);
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full),
                         "r"(bytes)
                         : "memory");
            if (bytes == 0) return;
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
                "[%0], [%1], %2, [%3], %4;"
                ::"r"(smem_u32(slot_codes(s))), "l"(src),
                "r"(bytes), "r"(full), "l"(evict_first)
                : "memory");
        };
        const int pre = has_first ? min(S, first.nsteps) : 0;
        if (lane == 0) {
            for (int st = 0; st < pre; ++st) {
                tail->slot_unit[st] = blockIdx.x;
                tail->slot_step[st] = st;
                tail->slot_meta[st] = slot_meta_pack(
                    first.width, min(kSlotGroups, first.ng - st * kSlotGroups), first.rows,
                    st == first.nsteps - 1);
                issue_codes(first, first_codes, st, st);
            }
        }
        w_issued = pre;
        asm volatile("griddepcontrol.wait;" ::: "memory");

        int u = blockIdx.x;
        uint32_t* work = a.counters + kWorkCounter;
        while (ok) {
            if (u >= total_units) {
                if (lane == 0) {
                    // the last CTA to run out of work resets the scheduler words
                    const uint32_t done = atomicAdd(a.counters + kDoneCounter, 1u);
                    if (done == gridDim.x - 1) {
                        a.counters[kWorkCounter] = 0u;
                        a.counters[kDoneCounter] = 0u;
                    }
                }
                break;
            }
            const Unit w = decode_unit<NT, kMode>(a, tail, u);
            const uint8_t* tile_codes = w.packed + packed_tile_base(a.K, w.tile);
            for (int st = 0; st < w.nsteps; ++st, ++step) {
                const int s = step % S;
                const uint32_t full = smem_u32(&tail->full[s]);
                if (step >= w_issued) {
                    if (step >= S && !warp_wait(smem_u32(&tail->empty[s]), ((step / S) - 1) & 1,
                                                abort, a.status)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        tail->slot_unit[s] = u;
                        tail->slot_step[s] = st;
                        tail->slot_meta[s] = slot_meta_pack(
                            w.width, min(kSlotGroups, w.ng - st * kSlotGroups), w.rows,
                            st == w.nsteps - 1);
                        issue_codes(w, tile_codes, st, step);
                    }
                    w_issued = step + 1;
                }
                // activations (valid rows only: the padding rows of an mma tile
                // keep whatever the slot held -- each batch row's outputs depend
                // only on its own row of x, and padding rows are never written),
                // scales, zero-points
                const int g0 = w.g_begin + st * kSlotGroups;
                const int ngs = min(kSlotGroups, w.g_begin + w.ng - g0);
                const uint32_t xbase = smem_u32(slot_x(s));
                const int p = lane & 15;
                for (int gl = 0; gl < ngs; ++gl)
                    for (int r = lane >> 4; r < w.rows; r += 2)
                        if (in_bounds(w.b0 + r < a.B && kGroup * (g0 + gl) + 8 * p + 8 <= a.K,
                                      a.status))
                            cp_async_16(
                                xbase + 16u * (((gl * 4 + (p & 3)) * kRows + r) * 4 + (p >> 2)),
                                a.x + (size_t)(w.b0 + r) * a.K + (size_t)kGroup * (g0 + gl) + 8 * p);
                const int gl = lane >> 4;
                if (gl < ngs && p < w.width / 8 &&
                    in_bounds(g0 + gl < a.K / kGroup && w.n0 + 8 * p + 8 <= a.N, a.status)) {
                    cp_async_16(smem_u32(slot_scales(s)) + 2u * (gl * kTileCols + 8 * p),
                                w.scales + (size_t)(g0 + gl) * a.N + w.n0 + 8 * p);
                    if (kHasZeros && in_bounds(w.n0 / 8 + p < a.zrow_words, a.status))
                        cp_async_4(smem_u32(slot_zeros(s)) + 4u * (gl * (kTileCols / 8) + p),
                                   w.zeros + (size_t)(g0 + gl) * a.zrow_words + w.n0 / 8 + p);
                }
                cp_async_arrive_noinc(full);
                issued = step + 1;
            }
            if (!ok) break;
            // next unit from the work counter (units [0, grid) are the fixed first ones)
            int next = 0;
            if (lane == 0) next = (int)gridDim.x + (int)atomicAdd(work, 1u);
            u = __shfl_sync(0xffffffffu, next, 0);  // the loop top checks it
        }
        // end marker for the consumers
        if (ok) {
            const int s = step % S;
            if (step < S || warp_wait(smem_u32(&tail->empty[s]), ((step / S) - 1) & 1, abort,
                                      a.status)) {
                if (lane == 0) {
                    tail->slot_unit[s] = -1;
                    mbar_arrive(smem_u32(&tail->full[s]));
                }
                cp_async_arrive_noinc(smem_u32(&tail->full[s]));
            }
        }
        // After an expired wait, every copy still in flight into the ring must
        // land before the CTA exits.  (On the normal path the consumers have
        // waited for every slot, and the end marker may already reuse a slot,
        // so there is nothing to drain.)
        for (int i = max(0, w_issued - S); !ok && i < w_issued; ++i) {
            const uint32_t full = smem_u32(&tail->full[i % S]);
            if (i >= issued) cp_async_arrive_noinc(full);
            wait_bounded(full, (i / S) & 1, abort, a.status);
        }
    } else if (warp <= kConsumerWarps) {
        // ---------------- consumers: warp cw owns columns 16cw .. 16cw+15 of the tile
        const int cw = warp - 1;
        const int gid = lane >> 2;  // mma group id: weight column within 8
        const int tig = lane & 3;   // which 32-row chunk of a group
        const int ca = 16 * cw + gid, cb = ca + 8;  // the two columns of this lane
        float acc[NT][4];
        int nunit = 0;  // units finished by this CTA
        for (int step = 0;; ++step) {
            const int s = step % S;
            if (!warp_wait(smem_u32(&tail->full[s]), (step / S) & 1, abort, a.status)) break;
            const int u = tail->slot_unit[s];
            const int st = tail->slot_step[s];
            const int buf = nunit & 1;
            if (u < 0) {
                // no more work: tell the epilogue warp
                if (nunit >= 2 && !warp_wait(smem_u32(&tail->res_empty[buf]), ((nunit >> 1) - 1) & 1,
                                             abort, a.status))
                    break;
                if (lane == 0) {
                    if (cw == 0) tail->res_unit[buf] = -1;
                    mbar_arrive(smem_u32(&tail->res_full[buf]));
                }
                break;
            }
            const int meta = tail->slot_meta[s];
            const int width = meta & 0xFF, ngs = (meta >> 8) & 0xF, rows = (meta >> 12) & 0xFF;
            const bool last = (meta >> 20) & 1;
            if (st == 0) {
#pragma unroll
                for (int bt = 0; bt < NT; ++bt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[bt][i] = 0.f;
            }
            const uint4* codes = reinterpret_cast<const uint4*>(slot_codes(s));
            const uint4* xs = slot_x(s);
            const uint16_t* sc = slot_scales(s);
            const uint32_t* zs = slot_zeros(s);
            const int cla = min(ca, width - 1), clb = min(cb, width - 1);
            const uint4* xq = xs + gid * 4 + tig;  // this lane's fragment column
#pragma unroll
            for (int gl = 0; gl < kSlotGroups; ++gl) {
                if (gl < ngs) {
                    // chunk 4(g0 + gl) + tig: its run is swizzled by 2 * tig
                    const uint4 qa = codes[(4 * gl + tig) * width + (cla ^ (2 * tig))];
                    const uint4 qb = codes[(4 * gl + tig) * width + (clb ^ (2 * tig))];
                    const float sa = Fmt::to_f32(sc[gl * kTileCols + cla]);
                    const float sb = Fmt::to_f32(sc[gl * kTileCols + clb]);
                    uint32_t za = Fmt::kSymZero2, zb = Fmt::kSymZero2;
                    if (kHasZeros) {
                        za = zero_pair<Fmt>((zs[gl * (kTileCols / 8) + (cla >> 3)] >> (4 * (cla & 7))) & 0xFu);
                        zb = zero_pair<Fmt>((zs[gl * (kTileCols / 8) + (clb >> 3)] >> (4 * (clb & 7))) & 0xFu);
                    }
                    const uint32_t wA[4] = {qa.x, qa.y, qa.z, qa.w};
                    const uint32_t wB[4] = {qb.x, qb.y, qb.z, qb.w};
                    float t[NT][4];  // this group's fp32 sums of (q - z) * x
#pragma unroll
                    for (int bt = 0; bt < NT; ++bt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) t[bt][i] = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint4 xf[NT];
#pragma unroll
                        for (int bt = 0; bt < NT; ++bt)
                            xf[bt] = xq[((gl * 4 + j) * kRows + bt * 8) * 4];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // step 2j + h: rows 4(2j+h) .. +3 of each lane's chunk
                            const uint32_t a0 = code_pair<Fmt>(wA[j], 2 * h, za);
                            const uint32_t a1 = code_pair<Fmt>(wB[j], 2 * h, zb);
                            const uint32_t a2 = code_pair<Fmt>(wA[j], 2 * h + 1, za);
                            const uint32_t a3 = code_pair<Fmt>(wB[j], 2 * h + 1, zb);
#pragma unroll
                            for (int bt = 0; bt < NT; ++bt)
                                if (bt * 8 < rows)  // warp-uniform: skip padding tiles
                                    mma_16816<Fmt>(t[bt], a0, a1, a2, a3, h ? xf[bt].z : xf[bt].x,
                                             h ? xf[bt].w : xf[bt].y);
                        }
                    }
#pragma unroll
                    for (int bt = 0; bt < NT; ++bt) {
                        acc[bt][0] = fmaf(sa, t[bt][0], acc[bt][0]);
                        acc[bt][1] = fmaf(sa, t[bt][1], acc[bt][1]);
                        acc[bt][2] = fmaf(sb, t[bt][2], acc[bt][2]);
                        acc[bt][3] = fmaf(sb, t[bt][3], acc[bt][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tail->empty[s]));

            if (last) {
                // unit finished: hand the accumulators to the epilogue warp
                if (nunit >= 2 && !warp_wait(smem_u32(&tail->res_empty[buf]), ((nunit >> 1) - 1) & 1,
                                             abort, a.status))
                    break;
                float* r = res + buf * (result_bytes<NT>() / 4);
#pragma unroll
                for (int bt = 0; bt < NT; ++bt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) r[((cw * NT + bt) * 4 + i) * 32 + lane] = acc[bt][i];
                __syncwarp();
                if (lane == 0) {
                    if (cw == 0) tail->res_unit[buf] = u;
                    mbar_arrive(smem_u32(&tail->res_full[buf]));
                }
                ++nunit;
            }
        }
    } else {
        // ---------------- epilogue warp: y, or split-K accumulation + conversion
        // Lane l owns columns 4l .. 4l+3 of the tile.
        const int c4 = 4 * lane;
        for (int k = 0;; ++k) {
            const int buf = k & 1;
            if (!warp_wait(smem_u32(&tail->res_full[buf]), (k >> 1) & 1, abort, a.status)) break;
            const int u = tail->res_unit[buf];
            if (u < 0) break;
            const Unit w = decode_unit<NT, kMode>(a, tail, u);
            const float* r = res + buf * (result_bytes<NT>() / 4);
            const bool mine = c4 < w.width;
            // element (column c, row b) of the unit lives at
            // r[((c/16 * NT + b/8) * 4 + i) * 32 + lane'], i = 2*((c%16)/8) + b%2,
            // lane' = 4*(c%8) + (b%8)/2
            auto elem = [&](int c, int b) {
                const int r16 = c & 15;
                const int i = ((r16 >> 3) << 1) | (b & 1);
                const int ln = (r16 & 7) * 4 + ((b & 7) >> 1);
                return r[(((c >> 4) * NT + (b >> 3)) * 4 + i) * 32 + ln];
            };
            for (int b = 0; b < w.rows && mine; ++b) {
                const float v0 = elem(c4, b), v1 = elem(c4 + 1, b), v2 = elem(c4 + 2, b),
                            v3 = elem(c4 + 3, b);
                const size_t off = (size_t)(w.b0 + b) * a.N + w.n0 + c4;
                if (!in_bounds(w.b0 + b < a.B && w.n0 + c4 + 4 <= a.N, a.status)) continue;
                if (a.split == 1) {
                    if constexpr (kMode == kFusedEpi)
                        epi_store4_fused(a.y, a.N, w.b0 + b, w.n0 + c4, v0, v1, v2, v3, a.epi);
                    else
                        store4<Fmt>(a.y + off, v0, v1, v2, v3);
                } else {
                    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                                 ::"l"(a.partial + off), "f"(v0), "f"(v1), "f"(v2), "f"(v3)
                                 : "memory");
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tail->res_empty[buf]));  // buffer free again
            if (a.split > 1) {
                // the last unit of this tile to arrive converts the fp32 sum to
                // bf16 and clears the accumulator for the next call.  Every lane
                // counts itself in with an acq_rel atomic, which orders its own
                // reductions before it -- no fence for the whole warp (measured:
                // down 14336 -> 4096 at B = 1 13.35 -> 12.33 us) -- and the lane
                // that sees 32 * split - 1 arrivals before it is the last.
                uint32_t* counter = a.counters + (size_t)w.bc * a.tiles + w.tile;
                if (!in_bounds((size_t)w.bc * a.tiles + w.tile < (size_t)kWorkCounter, a.status))
                    continue;
                uint32_t prev;
                asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                             : "=r"(prev)
                             : "l"(counter)
                             : "memory");
                if (__any_sync(0xffffffffu, prev == (uint32_t)(32 * a.split - 1))) {
                    // the last lane's acquire reaches the whole warp through the
                    // warp barrier; the fence orders the reads below after it
                    __syncwarp();
                    __threadfence();
                    for (int b0 = 0; b0 < w.rows && mine; b0 += 8) {
                        float4 v[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (b0 + j < w.rows &&
                                in_bounds(w.b0 + b0 + j < a.B && w.n0 + c4 + 4 <= a.N, a.status))
                                v[j] = __ldcg(reinterpret_cast<const float4*>(
                                    a.partial + (size_t)(w.b0 + b0 + j) * a.N + w.n0 + c4));
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (b0 + j < w.rows && w.b0 + b0 + j < a.B && w.n0 + c4 + 4 <= a.N) {
                                const size_t off = (size_t)(w.b0 + b0 + j) * a.N + w.n0 + c4;
                                if constexpr (kMode == kFusedEpi)
                                    epi_store4_fused(a.y, a.N, w.b0 + b0 + j, w.n0 + c4, v[j].x,
                                                     v[j].y, v[j].z, v[j].w, a.epi);
                                else
                                    store4<Fmt>(a.y + off, v[j].x, v[j].y, v[j].z, v[j].w);
                                __stcg(reinterpret_cast<float4*>(a.partial + off),
                                       make_float4(0.f, 0.f, 0.f, 0.f));
                            }
                        }
                    }
                    if (lane == 0) *counter = 0u;  // ready for the next call
                }
            }
        }
    }
    __syncthreads();
}

template <int NT, bool Z>
cudaError_t launch_t(const SkinnyPlan& p, Args a, cudaStream_t stream) {
    const size_t smem = (size_t)ring_slots<NT>() * slot_bytes<NT>() + 2 * result_bytes<NT>() +
                        sizeof(Tail);
    const void* kern =
        a.epi.f16            ? reinterpret_cast<const void*>(skinny_kernel<NT, Z, kPlain, F16>)
        : a.offsets != nullptr ? reinterpret_cast<const void*>(skinny_kernel<NT, Z, kGrouped, Bf16>)
        : a.epi.mode != 0    ? reinterpret_cast<const void*>(skinny_kernel<NT, Z, kFusedEpi, Bf16>)
                             : reinterpret_cast<const void*>(skinny_kernel<NT, Z, kPlain, Bf16>);
    cudaError_t err = set_smem_limit(kern, smem);
    if (err != cudaSuccess) return err;
    void* args[] = {&a};
    return launch_with_pdl(kern, dim3(p.grid), dim3(kThreads), smem, stream, args);
}

int ctas_per_sm(int nt) { return nt >= 4 ? 1 : (nt == 1 ? 3 : 2); }

}  // namespace

namespace {

// The K split for `chunks` batch chunks of a K x N layer (see plan_skinny).
void choose_split(SkinnyPlan& p, long long chunks, int K, int num_sms) {
    const int G = K / kGroup;
    const long long base = (long long)p.col_blocks * chunks;
    const long long slots = (long long)num_sms * ctas_per_sm(p.nt);
    int split = 1;
    while (split < G && split < 32 && base * split < slots) ++split;
    while (split < G && split < 32 && base * split < 3 * slots &&
           (G + split - 1) / split > 8)
        ++split;
    int gps = (G + split - 1) / split;
    split = (G + gps - 1) / gps;  // no empty units
    p.split = split;
    p.gps = gps;
}

}  // namespace

SkinnyPlan plan_skinny(int B, int K, int N, int num_sms) {
    SkinnyPlan p;
    p.nt = B <= 8 ? 1 : (B <= 16 ? 2 : 4);
    p.batch_chunks = (B + 8 * p.nt - 1) / (8 * p.nt);
    p.col_blocks = (N + kTileCols - 1) / kTileCols;
    // Units are handed out dynamically, so only their size matters: the K
    // split is the smallest that gives every CTA at least one unit (small
    // layers), and otherwise keeps units of a few ring slots so the tail
    // (the last units finishing) stays short, without multiplying the
    // split-K partial traffic.
    choose_split(p, p.batch_chunks, K, num_sms);
    const long long base = (long long)p.col_blocks * p.batch_chunks;
    if (base > kMaxCounters - 2) {
        p.split = 1;
        p.gps = K / kGroup;
    }
    const long long slots = (long long)num_sms * ctas_per_sm(p.nt);
    const long long units = base * p.split;
    p.units = (int)units;
    p.grid = (int)std::min<long long>(units, slots);
    return p;
}

SkinnyPlan plan_skinny_grouped(int T, int E, int max_rows, int K, int N, int num_sms) {
    SkinnyPlan p;
    // The batch tile follows the typical expert, not only the largest: a few
    // experts above the tile take two tiles (their weights are read twice),
    // which costs less than running every expert on a tile twice as tall
    // (measured, 128 experts top-8 at 64 tokens: mean 4 rows, max 9 --
    // 8-row tiles 57 us, 16-row tiles 63 us for the gate+up GEMM).
    const int typical = (T + E - 1) / E;
    p.nt = (max_rows <= 8 || typical <= 5) ? 1 : ((max_rows <= 16 || typical <= 10) ? 2 : 4);
    const int rows = 8 * p.nt;
    p.col_blocks = (N + kTileCols - 1) / kTileCols;
    // the chunks each expert's rows fill are only known on the device: size
    // the split for the typical count (every expert with rows, or the rows in
    // full chunks, whichever is more), and keep every possible chunk's
    // split-K counter inside the counter prefix
    const long long worst_chunks = std::min<long long>((long long)T, (long long)(T + rows - 1) / rows + E);
    const long long est_chunks = std::max<long long>((T + rows - 1) / rows, std::min(T, E));
    choose_split(p, est_chunks, K, num_sms);
    if (worst_chunks * p.col_blocks > kMaxCounters - 2) {
        p.split = 1;
        p.gps = K / kGroup;
    }
    p.batch_chunks = (int)worst_chunks;
    p.units = 0;  // counted on the device
    p.grid = num_sms * ctas_per_sm(p.nt);
    return p;
}

PlanResources skinny_resources(const SkinnyPlan& p) {
    PlanResources r{};
    const int nt = p.nt;
    const int slots = nt == 1 ? ring_slots<1>() : (nt == 2 ? ring_slots<2>() : ring_slots<4>());
    const size_t sb = nt == 1 ? slot_bytes<1>() : (nt == 2 ? slot_bytes<2>() : slot_bytes<4>());
    const size_t rb = nt == 1 ? result_bytes<1>() : (nt == 2 ? result_bytes<2>() : result_bytes<4>());
    r.smem = (size_t)slots * sb + 2 * rb + sizeof(Tail);
    r.ctas_per_sm = ctas_per_sm(nt);
    r.code_slots = slots;
    r.block_rows = kSlotGroups * kGroup;  // K rows per ring slot
    return r;
}

size_t skinny_workspace_bytes(const SkinnyPlan& p, int B, int N) {
    // counter prefix (also holds the scheduler's words) + one fp32 accumulator
    return p.split > 1 ? kCounterBytes + (size_t)B * N * sizeof(float) : kCounterBytes;
}

static cudaError_t launch_skinny_impl(const SkinnyPlan& p, const void* x, const void* packed,
                                      const void* scales, bool has_zeros, void* y, int B, int K,
                                      int N, void* workspace, unsigned int* status,
                                      const int* offsets, int E, const Epilogue& epi,
                                      cudaStream_t stream) {
    Args a;
    a.x = static_cast<const uint16_t*>(x);
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
    a.tiles = p.col_blocks;
    a.split = p.split;
    a.gps = p.gps;
    a.units = p.units;
    a.offsets = offsets;
    a.E = E;
    a.w_stride = packed_total_bytes(K, N, has_zeros);
    a.tag = a.packed + packed_tag_offset(K, N, has_zeros);
    a.code_bytes = code_bound_bytes(K, N);
    a.zrow_words = packed_zero_row_words(N);
    const BlobTag want = blob_tag(K, N, has_zeros);
    for (int i = 0; i < 4; ++i) a.tag_want[i] = want.w[i];
    a.s_stride = (size_t)(K / kGroup) * N;
    a.epi = epi;
    switch (p.nt * 2 + (has_zeros ? 1 : 0)) {
        case 2: return launch_t<1, false>(p, a, stream);
        case 3: return launch_t<1, true>(p, a, stream);
        case 4: return launch_t<2, false>(p, a, stream);
        case 5: return launch_t<2, true>(p, a, stream);
        case 8: return launch_t<4, false>(p, a, stream);
        case 9: return launch_t<4, true>(p, a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_skinny(const SkinnyPlan& p, const void* x, const void* packed,
                          const void* scales, bool has_zeros, void* y, int B, int K, int N,
                          void* workspace, unsigned int* status, const Epilogue& epi,
                          cudaStream_t stream) {
    return launch_skinny_impl(p, x, packed, scales, has_zeros, y, B, K, N, workspace, status,
                              nullptr, 0, epi, stream);
}

cudaError_t launch_skinny_grouped(const SkinnyPlan& p, const void* x, const int* offsets, int E,
                                  const void* packed, const void* scales, bool has_zeros,
                                  void* y, int T, int K, int N, void* workspace,
                                  unsigned int* status, cudaStream_t stream) {
    return launch_skinny_impl(p, x, packed, scales, has_zeros, y, T, K, N, workspace, status,
                              offsets, E, Epilogue{}, stream);
}

}  // namespace w4a16
