// launch.cuh -- internal launchers and planners behind the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace w4a16 {

constexpr int kGroup = 128;

inline size_t packed_code_bytes(int K, int N) { return (size_t)K * (size_t)N / 2; }
// Zero-point rows: N/8 words padded to a multiple of 4 (dequant.cuh).
inline size_t packed_zero_bytes(int K, int N) {
    return (size_t)(K / kGroup) * (size_t)(((N / 8) + 3) & ~3) * 4;
}
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Every packed blob ends with a 16-byte tag, written by the repack kernel:
// {kBlobMagic, layout version, K, N | has_zeros << 31}.  A GEMM kernel reads
// it once per CTA and records W4A16_ERR_UNSUPPORTED in the device status word
// if it does not describe the call (a blob from another layout version or
// another shape); w4a16_packed_check reads it on the host.
constexpr size_t kBlobTagBytes = 16;
constexpr uint32_t kBlobMagic = 0x70413457u;  // bytes 'W' '4' 'A' 'p'
constexpr uint32_t kBlobLayout = 4;           // W4A16_PACKED_LAYOUT
constexpr unsigned int kStatusBadBlob = 4;    // W4A16_ERR_UNSUPPORTED
inline size_t packed_tag_offset(int K, int N, bool has_zeros) {
    return packed_code_bytes(K, N) + (has_zeros ? packed_zero_bytes(K, N) : 0);
}
inline size_t packed_total_bytes(int K, int N, bool has_zeros) {
    return packed_tag_offset(K, N, has_zeros) + kBlobTagBytes;
}
// The tag a (K, N, has_zeros) call expects.
struct BlobTag {
    uint32_t w[4];
};
inline BlobTag blob_tag(int K, int N, bool has_zeros) {
    return BlobTag{{kBlobMagic, kBlobLayout, (uint32_t)K,
                    (uint32_t)N | (has_zeros ? 0x80000000u : 0u)}};
}

// Workspace layout shared by every kernel: a fixed prefix of counters
// (per-tile arrival counters and the small-batch kernel's work-scheduler
// words) and, after it, one fp32 accumulator [B][N] that split-K kernels add
// their partial sums into.  The caller zero-fills the workspace once; every
// call leaves all of it at zero again (the last CTA of a tile clears what it
// converted), so calls of different shapes can share one workspace.
constexpr int kMaxCounters = 16384;
constexpr size_t kCounterBytes = kMaxCounters * sizeof(uint32_t);
inline uint32_t* ws_counters(void* ws) { return static_cast<uint32_t*>(ws); }
inline float* ws_partials(void* ws) {
    return ws == nullptr ? nullptr
                         : reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes);
}

// Fused output epilogue (applied where the fp32 sums become bf16; see
// epilogue.cuh): flags of W4A16_EPI_* in w4a16.h.
constexpr int kEpiBias = 1;     // y = acc + bias[n]
constexpr int kEpiSiluMul = 2;  // y[b][j] = silu(acc[b][2j]) * acc[b][2j+1], y is [B][N/2]
struct Epilogue {
    const uint16_t* bias = nullptr;  // bf16 [N] with kEpiBias
    int mode = 0;
    // fp16 activations, scales and output (fmt16.cuh) instead of bf16; only
    // the plain epilogue (mode 0) has an fp16 form
    bool f16 = false;
};

// Extent of the packed codes the kernels' bounds checks compare against:
// packed_code_bytes(K, N), less the debug build's test cut
// (w4a16_debug_shrink_code_bound).
size_t code_bound_bytes(int K, int N);

// Sets a kernel's dynamic shared-memory limit once per (device, kernel):
// repeated calls with a size it already allows return at once.
cudaError_t set_smem_limit(const void* kernel, size_t bytes);

// Programmatic dependent launch: kernels may start (and prefetch weights)
// while the previous kernel on the stream finishes; they wait before reading
// activations or touching outputs and workspace.
cudaError_t launch_with_pdl(const void* func, dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, void** args);

cudaError_t launch_repack(const uint32_t* qweight, const uint32_t* qzeros, int K, int N,
                          void* packed, cudaStream_t stream);
cudaError_t launch_dequant_ref(const void* packed, const void* scales, bool has_zeros, void* w,
                               int K, int N, bool f16, cudaStream_t stream);
cudaError_t launch_quantize(const void* w, int K, int N, uint32_t* qweight, void* scales,
                            cudaStream_t stream);

// ---- small-batch streaming kernel (skinny.cu) ----
struct SkinnyPlan {
    int nt;            // n8 batch tiles per unit: 1, 2 or 4 (8, 16 or 32 rows)
    int batch_chunks;  // ceil(B / (8 * nt))
    int col_blocks;    // column tiles of 128
    int gps;           // groups of 128 rows per K split
    int split;         // number of K splits (1 = no workspace)
    int units;         // batch_chunks * col_blocks * split
    int grid;          // persistent CTAs
};
SkinnyPlan plan_skinny(int B, int K, int N, int num_sms);
size_t skinny_workspace_bytes(const SkinnyPlan& p, int B, int N);
struct PlanResources;
PlanResources skinny_resources(const SkinnyPlan& p);
// grouped (mixture-of-experts) variant: T rows of x sorted by expert, device
// offsets[E+1]; max_rows bounds one expert's rows (picks the batch tile)
SkinnyPlan plan_skinny_grouped(int T, int E, int max_rows, int K, int N, int num_sms);
cudaError_t launch_skinny_grouped(const SkinnyPlan& p, const void* x, const int* offsets, int E,
                                  const void* packed, const void* scales, bool has_zeros,
                                  void* y, int T, int K, int N, void* workspace,
                                  unsigned int* status, cudaStream_t stream);
cudaError_t launch_skinny(const SkinnyPlan& p, const void* x, const void* packed,
                          const void* scales, bool has_zeros, void* y, int B, int K, int N,
                          void* workspace, unsigned int* status, const Epilogue& epi,
                          cudaStream_t stream);

// ---- tcgen05 tensor-core kernel (tc_gemm.cu) ----
struct TcPlan {
    int bn;          // batch rows per CTA tile (MMA N): 16 .. 256, multiple of 16
    int batch_tiles; // ceil(B / bn)
    int col_tiles;   // ceil(N / 128)
    int kb_per_split;// 64-row K blocks per split
    int split;       // K splits (1 = no workspace)
    int grid;        // persistent CTAs
    int issuers;     // MMA-issuing threads, each with its own accumulator (1, 2, 4)
    int bufs;        // accumulator sets alternating between items (1, 2)
    int a_slots;     // dequantised weight tiles held in TMEM
    int nsub;        // 64-row K blocks per copy stage
    bool wide;       // more than 16 batch rows: the single-issuer kernel (tc_wide.cu)
    int sub;         // wide kernel: 64-row sub-blocks per block (1 or 2)
};
TcPlan plan_tc(int B, int K, int N, int num_sms);
// Launch resources of a plan (for w4a16_describe_plan): shared memory per CTA,
// the rings, the tensor-memory columns in use, the MMA-issuing threads.
struct PlanResources {
    size_t smem;
    int ctas_per_sm, issuers, acc_bufs, tile_slots, x_slots, code_slots, tmem_cols, block_rows;
};
PlanResources wide_resources(const TcPlan& p, int B, int N);
size_t tc_workspace_bytes(const TcPlan& p, int B, int N);
cudaError_t launch_tc(const TcPlan& p, const void* x, const void* packed, const void* scales,
                      bool has_zeros, void* y, int B, int K, int N, void* workspace,
                      unsigned int* status, const Epilogue& epi, cudaStream_t stream);
cudaError_t launch_tc_forced_timeout(const TcPlan& p, const void* x, const void* packed,
                                     const void* scales, bool has_zeros, void* y, int B, int K,
                                     int N, void* workspace, unsigned int* status, int wait_ms,
                                     cudaStream_t stream);
bool tc_available();
// wide batches (tc_wide.cu); plan_tc() routes there and launch_tc() follows the plan
TcPlan plan_tc_wide(int B, int K, int N, int num_sms);
cudaError_t launch_tc_wide(const TcPlan& p, const void* x, const void* packed,
                           const void* scales, bool has_zeros, void* y, int B, int K, int N,
                           void* workspace, unsigned int* status, int force_timeout_ms,
                           const Epilogue& epi, cudaStream_t stream);

// ---- W8A8-FP8 comparison path (fp8.cu) ----
struct Fp8Plan {
    int bn;           // batch rows per tile (MMA N): 16 .. 256, multiple of 16
    int batch_tiles;  // ceil(B / bn)
    int col_tiles;    // ceil(N / 128)
    int kb_per_split; // 128-row K blocks per split
    int split;        // K splits (1 = no workspace)
    int grid;         // persistent CTAs
};
Fp8Plan plan_fp8(int B, int K, int N, int num_sms);
size_t fp8_workspace_bytes(const Fp8Plan& p, int B, int N);
cudaError_t launch_fp8_quantize_rows(const void* x, int B, int K, void* xq, float* sx,
                                     cudaStream_t stream);
cudaError_t launch_fp8_quantize_cols(const void* w, int K, int N, void* wq, float* sw,
                                     cudaStream_t stream);
size_t fp8_packed_bytes(int K, int N);
cudaError_t launch_fp8_pack(const void* wq, int K, int N, void* packed, cudaStream_t stream);
cudaError_t launch_fp8_gemm(const Fp8Plan& p, const void* xq, const float* sx,
                            const void* wpacked, const float* sw, void* y, int B, int K, int N,
                            void* workspace, unsigned int* status, cudaStream_t stream);

// Validation + dispatch + launch shared by the C entry points (api.cu).
// Returns a w4a16_status value.
int gemm_entry(const void* x, const void* packed, const void* scales, int has_zeros, void* y,
               int B, int K, int N, int group_size, void* workspace, size_t ws_bytes, int path,
               void* stream);

}  // namespace w4a16
