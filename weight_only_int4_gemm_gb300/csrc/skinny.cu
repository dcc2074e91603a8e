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
//    the slot (one conflict-free 16-byte load per lane per chunk), decodes
//    them with the shared lop3 magic-number routine and feeds the bf16 pairs
//    as the A operand of warp-level m16n8k16 tensor-core products in which
//    the 16 rows are weight columns and the 8 columns batch rows (operands
//    swapped, so the batch pads only to 8).  The k order inside an mma is
//    free, so each lane's four k values per step are consecutive rows of its
//    own 32-row chunk; the activations are staged in exactly that fragment
//    order, which makes each fragment load one 16-byte read;
//  * work units are (batch chunk, column tile, K split); a K split writes
//    fp32 partials to the workspace and the last unit of a tile to finish
//    (arrival counter) sums them in a fixed order -- deterministic, no second
//    launch, no waiting on other CTAs;
//  * programmatic dependent launch: the first ring slots' weight copies are
//    issued before waiting for the previous kernel on the stream, so
//    consecutive layers' weight streams overlap.
// Every mbarrier wait is bounded; on expiry the kernel records
// W4A16_ERR_TIMEOUT in the device status word and returns.
#include <cuda_runtime.h>

#include <algorithm>

#include "dequant.cuh"
#include "launch.cuh"

namespace w4a16 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);  // 288
constexpr int kTileCols = kPackTileCols;             // 128 columns per tile
constexpr int kSlotGroups = 2;                       // 128-row groups per ring slot
constexpr uint32_t kSlotCodeBytes = kSlotGroups * 4 * kTileCols * 16;  // 16 KB
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr unsigned int kStatusTimeout = 7;           // W4A16_ERR_TIMEOUT

template <int NT> constexpr int ring_slots() { return NT >= 4 ? 6 : 4; }
template <int NT> constexpr uint32_t slot_x_bytes() { return kSlotGroups * 16 * 8 * NT * 16; }
constexpr uint32_t kSlotScaleBytes = kSlotGroups * kTileCols * 2;  // 512
constexpr uint32_t kSlotZeroBytes = kSlotGroups * kTileCols / 2;   // 128
template <int NT> constexpr uint32_t slot_bytes() {
    return kSlotCodeBytes + slot_x_bytes<NT>() + kSlotScaleBytes + kSlotZeroBytes;
}

struct Args {
    const uint16_t* x;
    const uint8_t* packed;
    const uint16_t* scales;
    const uint32_t* zeros;
    uint16_t* y;
    float* partial;      // [split][B][N]   (split > 1)
    uint32_t* counters;  // [batch_chunks][tiles] (fixed workspace prefix)
    unsigned int* status;
    int B, K, N;
    int tiles, split, gps, units;
};

struct Tail {
    uint64_t full[8];
    uint64_t empty[8];
    int abort;
    int is_last;
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

// 16- or 4-byte asynchronous copy global -> shared; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ void consumer_bar() {  // the 8 consumer warps only
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
}

// Work unit u -> (batch chunk, tile, split index).
struct Unit {
    int bc, tile, sk, g_begin, ng, n0, width, b0, rows;
};

template <int NT>
__device__ __forceinline__ Unit decode_unit(const Args& a, int u) {
    constexpr int kRows = 8 * NT;
    Unit w;
    w.sk = u % a.split;
    const int rest = u / a.split;
    w.tile = rest % a.tiles;
    w.bc = rest / a.tiles;
    const int G = a.K / kGroup;
    w.g_begin = w.sk * a.gps;
    w.ng = min(a.gps, G - w.g_begin);
    w.n0 = w.tile * kTileCols;
    w.width = packed_tile_width(a.N, w.tile);
    w.b0 = w.bc * kRows;
    w.rows = min(kRows, a.B - w.b0);
    return w;
}

// ------------------------------------------------------------ kernel

template <int NT, bool kHasZeros>
__global__ void __launch_bounds__(kThreads, 1) skinny_kernel(const Args a) {
    constexpr int kRows = 8 * NT;
    constexpr int S = ring_slots<NT>();
    extern __shared__ __align__(128) uint8_t smem[];
    Tail* tail = reinterpret_cast<Tail*>(smem + S * slot_bytes<NT>());
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
            // lane 0's expect-tx arrive + one cp.async arrive per producer lane
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&tail->full[s])),
                         "r"(33));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&tail->empty[s])),
                         "r"(kConsumerWarps));
        }
        tail->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ---------------- producer
        const int G = a.K / kGroup;
        (void)G;
        // pass 0: weight copies of the first S slots, before waiting for the
        // previous kernel; pass 1: everything else.
        int issued = 0;    // steps whose copies are all issued
        int w_issued = 0;  // steps whose code copy is issued
        for (int pass = 0; pass < 2; ++pass) {
            if (pass == 1) asm volatile("griddepcontrol.wait;" ::: "memory");
            int step = 0;
            bool stop = false;
            for (int u = blockIdx.x; u < a.units && !stop; u += gridDim.x) {
                const Unit w = decode_unit<NT>(a, u);
                const int nsteps = (w.ng + kSlotGroups - 1) / kSlotGroups;
                const uint8_t* tile_codes = a.packed + packed_tile_base(a.K, w.tile);
                for (int st = 0; st < nsteps; ++st, ++step) {
                    if (pass == 0 && step >= S) {
                        stop = true;
                        break;
                    }
                    const int s = step % S;
                    const int g0 = w.g_begin + st * kSlotGroups;
                    const int ngs = min(kSlotGroups, w.g_begin + w.ng - g0);
                    const uint32_t full = smem_u32(&tail->full[s]);
                    const bool weights_now = (pass == 0) || step >= S;
                    if (pass == 1 && step >= S) {
                        const bool ok = wait_bounded(smem_u32(&tail->empty[s]),
                                                     ((step / S) - 1) & 1, abort, a.status);
                        if (!__all_sync(0xffffffffu, ok)) {
                            stop = true;
                            break;
                        }
                    }
                    if (weights_now && lane == 0) {
                        const uint32_t bytes = (uint32_t)ngs * 4 * w.width * 16;
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                                     ::"r"(full), "r"(bytes)
                                     : "memory");
                        asm volatile(
                            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                            "[%0], [%1], %2, [%3];"
                            ::"r"(smem_u32(slot_codes(s))),
                            "l"(tile_codes + (size_t)(4 * g0) * w.width * 16), "r"(bytes),
                            "r"(full)
                            : "memory");
                    }
                    if (weights_now) w_issued = step + 1;
                    if (pass == 1) {
                        // activations in fragment order: piece (gl, r, p) of
                        // x[b0 + r][128*(g0+gl) + 8p .. +8], zero-filled past B
                        const uint32_t xbase = smem_u32(slot_x(s));
                        const int rows_alloc = ((w.rows + 7) / 8) * 8;
                        const int total = ngs * 16 * rows_alloc;
                        for (int e = lane; e < total; e += 32) {
                            const int p = e & 15;
                            const int r = (e >> 4) % rows_alloc;
                            const int gl = (e >> 4) / rows_alloc;
                            const bool valid = r < w.rows;
                            const uint16_t* src = a.x + (size_t)(w.b0 + (valid ? r : 0)) * a.K +
                                                  (size_t)kGroup * (g0 + gl) + 8 * p;
                            cp_async_16(xbase + 16u * (((gl * 4 + (p & 3)) * kRows + r) * 4 + (p >> 2)),
                                        src, valid ? 16u : 0u);
                        }
                        // scales: ngs rows of `width` bf16, 16-byte pieces
                        const int spr = w.width / 8;
                        for (int e = lane; e < ngs * spr; e += 32) {
                            const int gl = e / spr, j = e - gl * spr;
                            cp_async_16(smem_u32(slot_scales(s)) + 2u * (gl * kTileCols + 8 * j),
                                        a.scales + (size_t)(g0 + gl) * a.N + w.n0 + 8 * j, 16u);
                        }
                        if (kHasZeros) {
                            for (int e = lane; e < ngs * spr; e += 32) {
                                const int gl = e / spr, j = e - gl * spr;
                                cp_async_4(smem_u32(slot_zeros(s)) + 4u * (gl * (kTileCols / 8) + j),
                                           a.zeros + (size_t)(g0 + gl) * (a.N / 8) + w.n0 / 8 + j);
                            }
                        }
                        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];"
                                     ::"r"(full)
                                     : "memory");
                        issued = step + 1;
                    }
                }
            }
        }
        // Every copy into the ring must land before the CTA exits.  Steps whose
        // code copy went out early but whose other copies were never issued
        // (only after an expired wait) get their missing arrivals here.
        for (int i = max(0, w_issued - S); i < w_issued; ++i) {
            const uint32_t full = smem_u32(&tail->full[i % S]);
            if (i >= issued)
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(full)
                             : "memory");
            wait_bounded(full, (i / S) & 1, abort, a.status);
        }
    } else {
        // ---------------- consumers: warp cw owns columns 16cw .. 16cw+15 of the tile
        const int cw = warp - 1;
        const int gid = lane >> 2;  // mma group id: weight column within 8
        const int tig = lane & 3;   // which 32-row chunk of a group
        const int ca = 16 * cw + gid, cb = ca + 8;  // the two columns of this lane
        int step = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
            const Unit w = decode_unit<NT>(a, u);
            const int nsteps = (w.ng + kSlotGroups - 1) / kSlotGroups;
            float acc[NT][4];
#pragma unroll
            for (int bt = 0; bt < NT; ++bt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[bt][i] = 0.f;

            for (int st = 0; st < nsteps; ++st, ++step) {
                const int s = step % S;
                const bool landed =
                    wait_bounded(smem_u32(&tail->full[s]), (step / S) & 1, abort, a.status);
                if (!__all_sync(0xffffffffu, landed)) {
                    ok = false;
                    break;
                }
                const int ngs = min(kSlotGroups, w.ng - st * kSlotGroups);
                const uint4* codes = reinterpret_cast<const uint4*>(slot_codes(s));
                const uint4* xs = slot_x(s);
                const uint16_t* sc = slot_scales(s);
                const uint32_t* zs = slot_zeros(s);
#pragma unroll
                for (int gl = 0; gl < kSlotGroups; ++gl) {
                    if (gl < ngs) {
                        const uint4 qa = codes[(4 * gl + tig) * w.width + min(ca, w.width - 1)];
                        const uint4 qb = codes[(4 * gl + tig) * w.width + min(cb, w.width - 1)];
                        const uint32_t sa = scale_pair(sc[gl * kTileCols + ca]);
                        const uint32_t sb = scale_pair(sc[gl * kTileCols + cb]);
                        uint32_t za = kSymmetricZeroPair, zb = kSymmetricZeroPair;
                        if (kHasZeros) {
                            za = zero_pair((zs[gl * (kTileCols / 8) + (ca >> 3)] >> (4 * (ca & 7))) & 0xFu);
                            zb = zero_pair((zs[gl * (kTileCols / 8) + (cb >> 3)] >> (4 * (cb & 7))) & 0xFu);
                        }
                        const uint32_t wA[4] = {qa.x, qa.y, qa.z, qa.w};
                        const uint32_t wB[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint4 xf[NT];
#pragma unroll
                            for (int bt = 0; bt < NT; ++bt)
                                xf[bt] = xs[((gl * 4 + j) * kRows + bt * 8 + gid) * 4 + tig];
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                // step 2j + h: rows 4(2j+h) .. +3 of each lane's chunk
                                const uint32_t a0 = dequant_pair(wA[j], 2 * h, za, sa);
                                const uint32_t a1 = dequant_pair(wB[j], 2 * h, zb, sb);
                                const uint32_t a2 = dequant_pair(wA[j], 2 * h + 1, za, sa);
                                const uint32_t a3 = dequant_pair(wB[j], 2 * h + 1, zb, sb);
#pragma unroll
                                for (int bt = 0; bt < NT; ++bt)
                                    if (bt * 8 < w.rows)  // warp-uniform: skip padding tiles
                                        mma_bf16(acc[bt], a0, a1, a2, a3, h ? xf[bt].z : xf[bt].x,
                                                 h ? xf[bt].w : xf[bt].y);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];"
                                 ::"r"(smem_u32(&tail->empty[s]))
                                 : "memory");
            }
            if (!ok) break;

            // unit output: D row (gid or gid+8) = weight column, D column
            // (2*tig + (i & 1)) = batch row
#pragma unroll
            for (int bt = 0; bt < NT; ++bt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = (i & 2) ? cb : ca;
                    const int b = bt * 8 + 2 * tig + (i & 1);
                    if (c < w.width && b < w.rows) {
                        const size_t off = (size_t)(w.b0 + b) * a.N + w.n0 + c;
                        if (a.split == 1)
                            a.y[off] = f32_to_bf16_rn(acc[bt][i]);
                        else
                            a.partial[(size_t)w.sk * a.B * a.N + off] = acc[bt][i];
                    }
                }
            if (a.split > 1) {
                // the last unit of this tile to finish sums the partials in order
                __threadfence();
                consumer_bar();
                uint32_t* counter = a.counters + (size_t)w.bc * a.tiles + w.tile;
                if (threadIdx.x == 32) {
                    uint32_t prev;
                    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                                 : "=r"(prev)
                                 : "l"(counter)
                                 : "memory");
                    tail->is_last = (prev == (uint32_t)(a.split - 1));
                }
                consumer_bar();
                if (tail->is_last) {
                    __threadfence();
                    const int t = threadIdx.x - 32;
                    for (int e = t; e < w.rows * w.width; e += 32 * kConsumerWarps) {
                        const int r = e / w.width;
                        const int c = e - r * w.width;
                        const size_t off = (size_t)(w.b0 + r) * a.N + w.n0 + c;
                        float sum = 0.f;
                        for (int sk = 0; sk < a.split; ++sk)
                            sum += __ldcg(a.partial + (size_t)sk * a.B * a.N + off);
                        a.y[off] = f32_to_bf16_rn(sum);
                    }
                    if (t == 0) *counter = 0u;  // ready for the next call
                }
                consumer_bar();  // is_last is reused by the next unit
            }
        }
    }
    __syncthreads();
}

template <int NT, bool Z>
cudaError_t launch_t(const SkinnyPlan& p, Args a, cudaStream_t stream) {
    const size_t smem = (size_t)ring_slots<NT>() * slot_bytes<NT>() + sizeof(Tail);
    const void* kern = reinterpret_cast<const void*>(skinny_kernel<NT, Z>);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    void* args[] = {&a};
    return launch_with_pdl(kern, dim3(p.grid), dim3(kThreads), smem, stream, args);
}

int ctas_per_sm(int nt) { return nt >= 4 ? 1 : 2; }

}  // namespace

SkinnyPlan plan_skinny(int B, int K, int N, int num_sms) {
    SkinnyPlan p;
    p.nt = B <= 8 ? 1 : (B <= 16 ? 2 : 4);
    p.batch_chunks = (B + 8 * p.nt - 1) / (8 * p.nt);
    p.col_blocks = (N + kTileCols - 1) / kTileCols;
    const int G = K / kGroup;
    const long long base = (long long)p.col_blocks * p.batch_chunks;
    const int cps = ctas_per_sm(p.nt);
    // Choose the K split: estimated time = the busiest SM's groups plus a
    // fixed cost per unit (and per split, for the reduction).  CTA c takes
    // units c, c + grid, ...; SM m hosts CTAs m and m + num_sms.
    double best = 1e300;
    int best_split = 1;
    for (int split = 1; split <= std::min(G, 64); ++split) {
        const int gps = (G + split - 1) / split;
        if ((G + gps - 1) / gps != split) continue;  // no empty units
        if (split > 1 && base > kMaxCounters) break;
        const long long units = base * split;
        const long long grid = std::min<long long>(units, (long long)num_sms * cps);
        const long long q = units / grid, r = units % grid;
        auto n_of = [&](long long c) { return c < grid ? q + (c < r ? 1 : 0) : 0; };
        const long long sm_units = n_of(0) + (cps > 1 ? n_of(num_sms) : 0);
        const double per_unit = gps + (split > 1 ? 2.0 : 0.5);
        const double cost = (double)sm_units * per_unit / cps;
        if (cost < best - 1e-9) {
            best = cost;
            best_split = split;
        }
    }
    p.split = best_split;
    p.gps = (G + best_split - 1) / best_split;
    const long long units = base * p.split;
    p.units = (int)units;
    p.grid = (int)std::min<long long>(units, (long long)num_sms * cps);
    return p;
}

size_t skinny_workspace_bytes(const SkinnyPlan& p, int B, int N) {
    return split_workspace_bytes(p.split, B, N);
}

cudaError_t launch_skinny(const SkinnyPlan& p, const void* x, const void* packed,
                          const void* scales, bool has_zeros, void* y, int B, int K, int N,
                          void* workspace, unsigned int* status, cudaStream_t stream) {
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

}  // namespace w4a16
