// skinny.cu -- memory-bound small-batch W4A16 GEMM (decode, B <= ~32).
//
// At small B the layer is a weight stream: every weight is read once from HBM
// and used B times ("When quantization pays -- and when it does not", model of
// a decode step: the memory term W*b_w/beta dominates until the batch reaches
// the ridge).  The kernel therefore keeps packed codes out of shared memory
// entirely: each thread streams 16-byte chunks of packed codes straight into
// registers (non-allocating, read-once loads), decodes them with the shared
// lop3 magic-number routine, and feeds the bf16 pairs as the A operand of
// warp-level m16n8k16 tensor-core products in which the 16 rows are weight
// columns and the 8 columns are batch rows (the operands swapped, so the
// batch pads only to 8).  That keeps the CUDA-core work per weight at the
// decode alone.
//
// Latency, not bandwidth, is what a decode-sized layer fights (a 4096 x 4096
// layer is ~55 KB per SM), so the kernel keeps its dependency chain short:
//  * each warp puts its first round of weight loads in flight before anything
//    else, then triggers the next kernel on the stream (programmatic
//    dependent launch, so that kernel's weight stream overlaps this one's
//    tail) and only then waits for the previous kernel;
//  * the activations are staged with asynchronous zero-filling copies that
//    overlap the weight loads;
//  * K is split across the CTAs of one thread-block cluster (up to 16), whose
//    partial sums are combined on chip through distributed shared memory -- no
//    global workspace, no atomics, no second launch; the sum order is fixed, so
//    results are deterministic.
//
// Inside one mma the contraction order of k is free, so each lane's four k
// values per step are four consecutive rows of its own 32-row chunk; the
// activations are staged in shared memory in exactly that fragment order,
// which makes every fragment load one conflict-free 16-byte read.
#include <cuda_runtime.h>

#include <algorithm>

#include "dequant.cuh"
#include "launch.cuh"

namespace w4a16 {
namespace {

constexpr int kWarpsN = 2;                 // warps across columns (16 columns each)
constexpr int kWarpsK = 4;                 // warps across K groups
constexpr int kThreads = 32 * kWarpsN * kWarpsK;
constexpr int kColsPerCta = 16 * kWarpsN;  // 32
constexpr int kPrefetch = 4;               // groups of codes in flight per warp
constexpr int kMaxCluster = 16;            // CTAs along K sharing one column block

// Groups staged and streamed per round: 16 (8 when 32 batch rows are staged).
template <int NT>
constexpr int round_groups() { return NT >= 4 ? 8 : 16; }

struct Args {
    const uint16_t* x;
    const uint4* packed;
    const uint16_t* scales;
    const uint32_t* zeros;
    uint16_t* y;
    int B, K, N;
    int gps;    // groups of 128 rows per CTA
    int split;  // CTAs along K = cluster size
};

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src),
                 "r"(src_bytes)
                 : "memory");
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

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

template <int NT>
constexpr size_t xs_bytes() { return (size_t)round_groups<NT>() * 16 * 8 * NT * sizeof(uint4); }
template <int NT>
constexpr size_t red_bytes() { return (size_t)kWarpsK * kWarpsN * NT * 4 * 32 * sizeof(float); }

template <int NT, bool kHasZeros>
__global__ void __launch_bounds__(kThreads, 2) skinny_kernel(const Args a) {
    extern __shared__ uint4 smem[];
    constexpr int kRows = 8 * NT;                // batch rows per CTA
    constexpr int kRG = round_groups<NT>();      // groups per round
    constexpr int kPerWarp = kRG / kWarpsK;      // groups per warp per round (<= kPrefetch)
    static_assert(kPerWarp <= kPrefetch, "round larger than the prefetch registers");

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int wn = warp % kWarpsN;
    const int wk = warp / kWarpsN;
    const int gid = lane >> 2;  // mma group id: weight column within 8
    const int tig = lane & 3;   // thread in group: which 32-row chunk of a group

    const int G = a.K / kGroup;
    const int g_begin = blockIdx.y * a.gps;
    const int ng = max(0, min(a.gps, G - g_begin));
    const int b0 = blockIdx.z * kRows;
    const int rows = min(kRows, a.B - b0);
    const int n_cta = blockIdx.x * kColsPerCta;
    const int n0 = n_cta + wn * 16;
    const int na = min(n0 + gid, a.N - 1);
    const int nb = min(n0 + gid + 8, a.N - 1);
    const int rounds = (ng + kRG - 1) / kRG;

    uint4* xs = smem;
    float* red = reinterpret_cast<float*>(reinterpret_cast<char*>(smem) + xs_bytes<NT>());

    // Weight registers for one round: group gl = round*kRG + u*kWarpsK + wk.
    uint4 wa[kPerWarp], wb[kPerWarp];
    uint32_t sa[kPerWarp], sb[kPerWarp], za[kPerWarp], zb[kPerWarp];
    auto load_round = [&](int rd) {
#pragma unroll
        for (int u = 0; u < kPerWarp; ++u) {
            const int gl = rd * kRG + u * kWarpsK + wk;
            if (gl < ng) {
                const int g = g_begin + gl;
                const size_t c = (size_t)(4 * g + tig) * a.N;
                wa[u] = ld_stream(a.packed + c + na);
                wb[u] = ld_stream(a.packed + c + nb);
                sa[u] = scale_pair(__ldg(a.scales + (size_t)g * a.N + na));
                sb[u] = scale_pair(__ldg(a.scales + (size_t)g * a.N + nb));
                if (kHasZeros) {
                    za[u] = zero_pair(load_zero(a.zeros, a.N, g, na));
                    zb[u] = zero_pair(load_zero(a.zeros, a.N, g, nb));
                } else {
                    za[u] = zb[u] = kSymmetricZeroPair;
                }
            }
        }
    };

    // 1. First round of weights in flight; then let the next kernel start and
    //    wait for the previous one (x and y may be its output / input).
    load_round(0);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float acc[NT][4];
#pragma unroll
    for (int bt = 0; bt < NT; ++bt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[bt][i] = 0.f;

    for (int rd = 0; rd < rounds; ++rd) {
        const int rg0 = rd * kRG;
        const int rng = min(kRG, ng - rg0);
        if (rd > 0) {
            __syncthreads();  // everyone is done reading the previous round's x
            load_round(rd);
        }
        // 2. Stage x[b0 .. b0+kRows)[round's groups] in fragment order:
        //    entry ((gl*4 + m)*kRows + r)*4 + t = x[b0+r][128*g + 32t + 8m .. +8].
        {
            const int pieces_per_row = rng * 16;
            const int total = pieces_per_row * kRows;
            for (int e = threadIdx.x; e < total; e += kThreads) {
                const int r = e / pieces_per_row;
                const int p = e - r * pieces_per_row;
                const int gl = p >> 4;
                const int within = p & 15;  // 8-row piece within the group
                const bool valid = r < rows;
                const uint16_t* src = a.x + (size_t)(b0 + (valid ? r : 0)) * a.K +
                                      (size_t)kGroup * (g_begin + rg0 + gl) + 8 * within;
                cp_async_16(&xs[((gl * 4 + (within & 3)) * kRows + r) * 4 + (within >> 2)], src,
                            valid ? 16u : 0u);
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
        }
        __syncthreads();

        // 3. Decode and multiply this round's groups.
#pragma unroll
        for (int u = 0; u < kPerWarp; ++u) {
            const int gl = u * kWarpsK + wk;  // within the round
            if (gl < rng) {
                const uint32_t wA[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
                const uint32_t wB[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 xf[NT];
#pragma unroll
                    for (int bt = 0; bt < NT; ++bt)
                        xf[bt] = xs[((gl * 4 + j) * kRows + bt * 8 + gid) * 4 + tig];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // step s = 2j + h: rows 4s .. 4s+3 of each lane's chunk
                        const uint32_t a0 = dequant_pair(wA[j], 2 * h, za[u], sa[u]);
                        const uint32_t a1 = dequant_pair(wB[j], 2 * h, zb[u], sb[u]);
                        const uint32_t a2 = dequant_pair(wA[j], 2 * h + 1, za[u], sa[u]);
                        const uint32_t a3 = dequant_pair(wB[j], 2 * h + 1, zb[u], sb[u]);
#pragma unroll
                        for (int bt = 0; bt < NT; ++bt)
                            if (bt * 8 < rows)  // warp-uniform: skip all-padding tiles
                                mma_bf16(acc[bt], a0, a1, a2, a3, h ? xf[bt].z : xf[bt].x,
                                         h ? xf[bt].w : xf[bt].y);
                    }
                }
            }
        }
    }

    // 4. Every warp's partial tile into shared memory, lane-minor.
#pragma unroll
    for (int bt = 0; bt < NT; ++bt)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            red[((warp * NT + bt) * 4 + i) * 32 + lane] = acc[bt][i];
    if (a.split > 1)
        cluster_sync_all();  // partials of every CTA of the cluster are visible
    else
        __syncthreads();

    // 5. Sum over the K-warps of every CTA of the cluster in a fixed order;
    //    output element e (column-minor) is finished by cluster rank e % split.
    uint32_t rank = 0;
    if (a.split > 1) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int cols = min(kColsPerCta, a.N - n_cta);
    for (int e = threadIdx.x * a.split + (int)rank; e < kColsPerCta * rows; e += kThreads * a.split) {
        const int nl = e % kColsPerCta;
        const int bl = e / kColsPerCta;
        if (nl >= cols) continue;
        const int w_n = nl >> 4, r16 = nl & 15;
        const int bt = bl >> 3, b8 = bl & 7;
        const int i = ((r16 >> 3) << 1) | (b8 & 1);
        const int ln = (r16 & 7) * 4 + (b8 >> 1);
        float s = 0.f;
        for (int q = 0; q < a.split; ++q) {
#pragma unroll
            for (int k = 0; k < kWarpsK; ++k) {
                const float* src = &red[(((k * kWarpsN + w_n) * NT + bt) * 4 + i) * 32 + ln];
                s += a.split > 1 ? ld_cluster_f32(src, (uint32_t)q) : *src;
            }
        }
        a.y[(size_t)(b0 + bl) * a.N + n_cta + nl] = f32_to_bf16_rn(s);
    }
    if (a.split > 1) cluster_sync_all();  // keep shared memory alive for remote readers
}

template <int NT, bool Z>
cudaError_t launch_t(const SkinnyPlan& p, Args a, cudaStream_t stream) {
    const size_t smem = xs_bytes<NT>() + red_bytes<NT>();
    const void* kern = reinterpret_cast<const void*>(skinny_kernel<NT, Z>);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    if (p.split > 8) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.col_blocks, p.split, p.batch_chunks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = p.split;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void* args[] = {&a};
    return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace

SkinnyPlan plan_skinny(int B, int K, int N, int num_sms) {
    SkinnyPlan p;
    p.nt = B <= 8 ? 1 : (B <= 16 ? 2 : 4);
    p.batch_chunks = (B + 8 * p.nt - 1) / (8 * p.nt);
    p.col_blocks = (N + kColsPerCta - 1) / kColsPerCta;
    const int G = K / kGroup;
    const int rg = p.nt >= 4 ? 8 : 16;
    const long long base = (long long)p.col_blocks * p.batch_chunks;
    const long long slots = 2LL * num_sms;  // two CTAs per SM (launch bounds)
    // choose the cluster size (K split) minimising waves x per-CTA time, the
    // per-CTA time being its groups plus a fixed cost per round and per CTA
    double best = 1e300;
    int best_split = std::min(G, kMaxCluster);
    for (int split = 1; split <= std::min(G, kMaxCluster); ++split) {
        const int gps = (G + split - 1) / split;
        if ((G + gps - 1) / gps != split) continue;  // no empty CTAs
        const long long ctas = base * split;
        const long long waves = (ctas + slots - 1) / slots;
        const int rounds = (gps + rg - 1) / rg;
        const double cost = (double)waves * (gps + 6.0 * rounds + 6.0) + 0.25 * split;
        if (cost < best - 1e-9) {
            best = cost;
            best_split = split;
        }
    }
    p.split = best_split;
    p.gps = (G + best_split - 1) / best_split;
    return p;
}

size_t skinny_workspace_bytes(const SkinnyPlan&, int, int) { return 0; }

cudaError_t launch_skinny(const SkinnyPlan& p, const void* x, const void* packed,
                          const void* scales, bool has_zeros, void* y, int B, int K, int N,
                          void* workspace, cudaStream_t stream) {
    (void)workspace;  // split-K is reduced on chip (cluster shared memory)
    Args a;
    a.x = static_cast<const uint16_t*>(x);
    a.packed = static_cast<const uint4*>(packed);
    a.scales = static_cast<const uint16_t*>(scales);
    a.zeros = reinterpret_cast<const uint32_t*>(static_cast<const char*>(packed) +
                                                packed_code_bytes(K, N));
    a.y = static_cast<uint16_t*>(y);
    a.B = B;
    a.K = K;
    a.N = N;
    a.gps = p.gps;
    a.split = p.split;
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
