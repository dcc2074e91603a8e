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
// The K dimension is split three ways: the four lanes of a quad each own one
// 32-row chunk of a 128-row group; the warps of a CTA take alternate groups
// (reduced through shared memory); CTAs take consecutive group ranges and
// combine through fp32 partials in the workspace, the last CTA to arrive at a
// column block summing them in a fixed order (deterministic, no second
// launch, no waiting).
//
// Inside one mma the contraction order of k is free, so each lane's four k
// values per step are four consecutive rows of its own chunk; the activations
// are staged in shared memory in exactly that fragment order, which makes
// every fragment load one conflict-free 16-byte read.
#include <cuda_runtime.h>

#include <algorithm>

#include "dequant.cuh"
#include "launch.cuh"

namespace w4a16 {
namespace {

constexpr int kWarpsN = 4;                 // warps across columns
constexpr int kWarpsK = 2;                 // warps across K groups
constexpr int kThreads = 32 * kWarpsN * kWarpsK;
constexpr int kColsPerCta = 16 * kWarpsN;  // 64
constexpr int kPrefetch = 4;               // groups of codes in flight per warp
constexpr int kMaxGps = kWarpsK * kPrefetch;  // groups per CTA = one round of loads
constexpr int kMaxRowsTimesGps = 128;      // caps the staged x slice at 64 KB

struct Args {
    const uint16_t* x;
    const uint4* packed;
    const uint16_t* scales;
    const uint32_t* zeros;
    uint16_t* y;
    float* partial;      // [split][B][N]
    uint32_t* counters;  // [batch_chunks][col_blocks] (fixed workspace prefix)
    int B, K, N;
    int gps, split;
};

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
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

template <int NT, bool kHasZeros>
__global__ void __launch_bounds__(kThreads, 2) skinny_kernel(const Args a) {
    extern __shared__ uint4 smem[];
    constexpr int kRows = 8 * NT;  // batch rows per CTA pass

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int wn = warp % kWarpsN;
    const int wk = warp / kWarpsN;
    const int gid = lane >> 2;  // mma group id: weight column within 8
    const int tig = lane & 3;   // thread in group: which 32-row chunk of a group

    const int G = a.K / kGroup;
    const int g_begin = blockIdx.y * a.gps;
    const int ng = min(a.gps, G - g_begin);
    const int b0 = blockIdx.z * kRows;
    const int rows = min(kRows, a.B - b0);
    const int n_cta = blockIdx.x * kColsPerCta;
    const int n0 = n_cta + wn * 16;
    const int na = min(n0 + gid, a.N - 1);
    const int nb = min(n0 + gid + 8, a.N - 1);

    // 1. Weights, scales and zero-points do not depend on the previous kernel:
    //    put this warp's first round of loads in flight before anything else.
    uint4 wa[kPrefetch], wb[kPrefetch];
    uint32_t sa[kPrefetch], sb[kPrefetch], za[kPrefetch], zb[kPrefetch];
    auto load_round = [&](int gl0) {
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int gl = gl0 + u * kWarpsK;
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
    load_round(wk);

    // 2. Let the next kernel on the stream start its own weight stream, then
    //    wait for the previous one before reading x or touching outputs.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // 3. Stage x[b0 .. b0+kRows)[group range] in fragment order:
    //    entry ((gl*4 + m)*kRows + r)*4 + t = x[b0+r][128*(g_begin+gl) + 32t + 8m .. +8].
    uint4* xs = smem;
    {
        const int pieces_per_row = ng * 16;
        const int total = pieces_per_row * kRows;
        for (int e = threadIdx.x; e < total; e += kThreads) {
            const int r = e / pieces_per_row;
            const int p = e - r * pieces_per_row;
            const int gl = p >> 4;
            const int within = p & 15;  // 8-row piece within the group
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows)
                v = __ldg(reinterpret_cast<const uint4*>(
                    a.x + (size_t)(b0 + r) * a.K + (size_t)kGroup * (g_begin + gl) + 8 * within));
            xs[((gl * 4 + (within & 3)) * kRows + r) * 4 + (within >> 2)] = v;
        }
    }
    __syncthreads();

    // 4. Decode and multiply, one round of prefetched groups at a time.
    float acc[NT][4];
#pragma unroll
    for (int bt = 0; bt < NT; ++bt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[bt][i] = 0.f;

    for (int gl0 = wk; gl0 < ng; gl0 += kWarpsK * kPrefetch) {
        if (gl0 != wk) load_round(gl0);
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int gl = gl0 + u * kWarpsK;
            if (gl < ng) {
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

    // 5. Reduce the K-warps through shared memory (fixed order).
    float* red = reinterpret_cast<float*>(smem + (size_t)a.gps * 16 * kRows);
    if (kWarpsK > 1) {
        if (wk > 0) {
#pragma unroll
            for (int bt = 0; bt < NT; ++bt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    red[(((wk - 1) * kWarpsN + wn) * NT * 4 + bt * 4 + i) * 32 + lane] = acc[bt][i];
        }
        __syncthreads();
        if (wk == 0) {
#pragma unroll
            for (int w = 1; w < kWarpsK; ++w)
#pragma unroll
                for (int bt = 0; bt < NT; ++bt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        acc[bt][i] += red[(((w - 1) * kWarpsN + wn) * NT * 4 + bt * 4 + i) * 32 + lane];
        }
    }

    // 6. Output: D row (gid or gid+8) is a weight column, D column
    //    (2*tig + (i & 1)) a batch row.
    if (wk == 0) {
#pragma unroll
        for (int bt = 0; bt < NT; ++bt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int n = n0 + gid + ((i & 2) ? 8 : 0);
                const int b = b0 + bt * 8 + 2 * tig + (i & 1);
                if (n < a.N && b < a.B) {
                    if (a.split == 1)
                        a.y[(size_t)b * a.N + n] = f32_to_bf16_rn(acc[bt][i]);
                    else
                        a.partial[((size_t)blockIdx.y * a.B + b) * a.N + n] = acc[bt][i];
                }
            }
    }
    if (a.split == 1) return;

    // 7. Last CTA of this column block sums the split partials in order.
    __shared__ int s_is_last;
    __threadfence();
    __syncthreads();
    uint32_t* counter = a.counters + (size_t)blockIdx.z * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0) {
        uint32_t prev;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(counter)
                     : "memory");
        s_is_last = (prev == (uint32_t)(a.split - 1));
    }
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    const int cols = min(kColsPerCta, a.N - n_cta);
    for (int e = threadIdx.x; e < rows * cols; e += kThreads) {
        const int r = e / cols;
        const int cc = e - r * cols;
        const size_t off = (size_t)(b0 + r) * a.N + n_cta + cc;
        float s = 0.f;
        for (int sk = 0; sk < a.split; ++sk)
            s += __ldcg(a.partial + (size_t)sk * a.B * a.N + off);
        a.y[off] = f32_to_bf16_rn(s);
    }
    if (threadIdx.x == 0) *counter = 0u;  // ready for the next call
}

template <int NT>
size_t smem_for(int gps) {
    return (size_t)gps * 16 * 8 * NT * sizeof(uint4) +
           (size_t)(kWarpsK - 1) * kWarpsN * NT * 4 * 32 * sizeof(float);
}

template <int NT, bool Z>
cudaError_t launch_t(const SkinnyPlan& p, Args a, cudaStream_t stream) {
    const size_t smem = smem_for<NT>(p.gps);
    const void* kern = reinterpret_cast<const void*>(skinny_kernel<NT, Z>);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    void* args[] = {&a};
    return launch_with_pdl(kern, dim3(p.col_blocks, p.split, p.batch_chunks), dim3(kThreads),
                           smem, stream, args);
}

int resident_ctas_per_sm(int nt) {
    // registers bound the residency; two CTAs per SM is what the kernel is
    // built for (launch bounds), one when the staged slice is large
    return nt >= 4 ? 1 : 2;
}

}  // namespace

SkinnyPlan plan_skinny(int B, int K, int N, int num_sms) {
    SkinnyPlan p;
    p.nt = B <= 8 ? 1 : (B <= 16 ? 2 : 4);
    p.batch_chunks = (B + 8 * p.nt - 1) / (8 * p.nt);
    p.col_blocks = (N + kColsPerCta - 1) / kColsPerCta;
    const int G = K / kGroup;
    const int cap = std::max(1, std::min(kMaxGps, kMaxRowsTimesGps / (8 * p.nt)));
    const long long base = (long long)p.col_blocks * p.batch_chunks;
    const long long slots = (long long)num_sms * resident_ctas_per_sm(p.nt);
    // choose groups per CTA minimising (waves x per-CTA time), per-CTA time
    // being its groups plus a fixed cost (launch, staging, reduction)
    double best = 1e300;
    int best_gps = std::min(cap, G);
    for (int gps = std::min(cap, G); gps >= 1; --gps) {
        const int split = (G + gps - 1) / gps;
        if (split > 1 && base > kMaxCounters) break;
        const long long ctas = base * split;
        const long long waves = (ctas + slots - 1) / slots;
        const double cost = (double)waves * (gps + 2.0) + (split > 1 ? 0.5 : 0.0);
        if (cost < best - 1e-9) {
            best = cost;
            best_gps = gps;
        }
    }
    p.gps = best_gps;
    p.split = (G + best_gps - 1) / best_gps;
    if (p.split > 1 && base > kMaxCounters) {  // no counters to spare: one CTA per column block
        p.gps = G;
        p.split = 1;
    }
    return p;
}

size_t skinny_workspace_bytes(const SkinnyPlan& p, int B, int N) {
    return split_workspace_bytes(p.split, B, N);
}

cudaError_t launch_skinny(const SkinnyPlan& p, const void* x, const void* packed,
                          const void* scales, bool has_zeros, void* y, int B, int K, int N,
                          void* workspace, cudaStream_t stream) {
    Args a;
    a.x = static_cast<const uint16_t*>(x);
    a.packed = static_cast<const uint4*>(packed);
    a.scales = static_cast<const uint16_t*>(scales);
    a.zeros = reinterpret_cast<const uint32_t*>(static_cast<const char*>(packed) +
                                                packed_code_bytes(K, N));
    a.y = static_cast<uint16_t*>(y);
    a.partial = ws_partials(workspace);
    a.counters = ws_counters(workspace);
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
