// api.cu -- the C ABI: host-side validation, path selection and launches.
// Nothing here allocates device memory or synchronises (except
// w4a16_device_status, which is documented to).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "w4a16.h"
#include "w8a8_fp8.h"
#include "checks.cuh"
#include "launch.cuh"

namespace w4a16 {
namespace {

constexpr int kMaxK = 1 << 20;
constexpr int kMaxN = 1 << 22;
constexpr int kMaxB = 1 << 20;

__device__ unsigned int g_device_status;  // tensor-core kernel's timeout flag

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool shape_ok(int K, int N) {
    return K > 0 && N > 0 && K % kGroup == 0 && N % 8 == 0 && K <= kMaxK && N <= kMaxN;
}

struct DeviceInfo {
    int sms = 0;
    int major = 0, minor = 0;
};

DeviceInfo device_info() {
    static std::mutex mu;
    static std::unordered_map<int, DeviceInfo> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DeviceInfo{};
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    DeviceInfo info;
    cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&info.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&info.minor, cudaDevAttrComputeCapabilityMinor, dev);
    cache[dev] = info;
    return info;
}

// Device address of the status word on the current device (cached per device).
unsigned int* device_status_word() {
    static std::mutex mu;
    static std::unordered_map<int, unsigned int*> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    unsigned int* p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_device_status) != cudaSuccess)
        return nullptr;
    cache[dev] = p;
    return p;
}

int num_sms() {
    const int s = device_info().sms;
    return s > 0 ? s : 152;
}

// Per-shape plan cache: the planners are pure functions of (B, K, N, SM
// count), and an eager caller repeats the same few shapes; one mutex guards
// it (the library is otherwise stateless).
struct PlanKey {
    int dev, B, K, N;
    bool operator==(const PlanKey& o) const {
        return dev == o.dev && B == o.B && K == o.K && N == o.N;
    }
};
struct PlanKeyHash {
    size_t operator()(const PlanKey& k) const {
        return ((size_t)k.dev * 1000003u ^ (size_t)k.B * 7919u) * 131u ^ (size_t)k.K * 31u ^
               (size_t)k.N;
    }
};
constexpr size_t kMaxCachedPlans = 4096;

template <typename Plan, typename Make>
Plan cached_plan(std::unordered_map<PlanKey, Plan, PlanKeyHash>& cache, std::mutex& mu, int B,
                 int K, int N, Make make) {
    int dev = 0;
    cudaGetDevice(&dev);
    const PlanKey key{dev, B, K, N};
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const Plan p = make();
    if (cache.size() >= kMaxCachedPlans) cache.clear();  // bounded: many distinct shapes
    cache.emplace(key, p);
    return p;
}

SkinnyPlan skinny_plan(int B, int K, int N) {
    static std::mutex mu;
    static std::unordered_map<PlanKey, SkinnyPlan, PlanKeyHash> cache;
    return cached_plan(cache, mu, B, K, N, [&] { return plan_skinny(B, K, N, num_sms()); });
}

TcPlan tc_plan(int B, int K, int N) {
    static std::mutex mu;
    static std::unordered_map<PlanKey, TcPlan, PlanKeyHash> cache;
    return cached_plan(cache, mu, B, K, N, [&] { return plan_tc(B, K, N, num_sms()); });
}

// Batch above which the tensor-core kernel takes over from the split-K
// kernel.  Measured on GB300 (decoder-layer shapes): the mma.sync kernel is
// faster up to 8 rows, the two are even at 16, and from 17 rows (where the
// mma.sync kernel needs 32-row batch tiles) the tensor-core kernel is 1.7x
// faster.
constexpr int kSkinnyMaxB = 16;
constexpr int kMaxGroupedExperts = 256;

// Override of the automatic choice for tests and ablations:
// W4A16_FORCE_PATH=skinny (or 0) / tcgen05 (or 1), read once per process; a
// forced tensor-core path is ignored on a device without it.
int forced_path() {
    static const int v = [] {
        const char* e = std::getenv("W4A16_FORCE_PATH");
        if (e == nullptr) return (int)W4A16_PATH_AUTO;
        if (!std::strcmp(e, "skinny") || !std::strcmp(e, "0")) return (int)W4A16_PATH_SKINNY;
        if (!std::strcmp(e, "tcgen05") || !std::strcmp(e, "1")) return (int)W4A16_PATH_TCGEN05;
        return (int)W4A16_PATH_AUTO;
    }();
    return v;
}

int choose_path(int B, int K, int N) {
    (void)K;
    (void)N;
    const int forced = forced_path();
    if (forced == W4A16_PATH_SKINNY) return W4A16_PATH_SKINNY;
    if (forced == W4A16_PATH_TCGEN05 && tc_available()) return W4A16_PATH_TCGEN05;
    if (B <= kSkinnyMaxB || !tc_available()) return W4A16_PATH_SKINNY;
    return W4A16_PATH_TCGEN05;
}

size_t path_workspace(int path, int B, int K, int N) {
    if (path == W4A16_PATH_SKINNY)
        return skinny_workspace_bytes(skinny_plan(B, K, N), B, N);
    return tc_workspace_bytes(tc_plan(B, K, N), B, N);
}

w4a16_status from_cuda(cudaError_t e) { return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA; }

w4a16_status gemm_impl(const void* x, const void* packed, const void* scales, int has_zeros,
                       void* y, int B, int K, int N, int group_size, void* workspace,
                       size_t ws_bytes, int path, void* stream, int forced_timeout_ms = 0,
                       const Epilogue& epi = Epilogue{}) {
    if (group_size != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (!shape_ok(K, N) || B < 1 || B > kMaxB) return W4A16_ERR_SHAPE;
    if (!x || !packed || !scales || !y) return W4A16_ERR_NULL;
    if (!aligned16(x) || !aligned16(packed) || !aligned16(scales) || !aligned16(y))
        return W4A16_ERR_ALIGN;
    if (path == W4A16_PATH_AUTO) path = choose_path(B, K, N);
    if (path != W4A16_PATH_SKINNY && path != W4A16_PATH_TCGEN05) return W4A16_ERR_UNSUPPORTED;
    if (path == W4A16_PATH_TCGEN05 && !tc_available()) return W4A16_ERR_UNSUPPORTED;
    const size_t need = path_workspace(path, B, K, N);
    if (need > 0) {
        if (workspace == nullptr) return W4A16_ERR_NULL;
        if (!aligned16(workspace)) return W4A16_ERR_ALIGN;
        if (ws_bytes < need) return W4A16_ERR_WORKSPACE;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* status = device_status_word();
    if (status == nullptr) return W4A16_ERR_CUDA;
    if (path == W4A16_PATH_SKINNY)
        return from_cuda(launch_skinny(skinny_plan(B, K, N), x, packed, scales,
                                       has_zeros != 0, y, B, K, N, workspace, status, epi, s));
    if (forced_timeout_ms > 0)
        return from_cuda(launch_tc_forced_timeout(tc_plan(B, K, N), x, packed, scales,
                                                  has_zeros != 0, y, B, K, N, workspace, status,
                                                  forced_timeout_ms, s));
    return from_cuda(launch_tc(tc_plan(B, K, N), x, packed, scales, has_zeros != 0,
                               y, B, K, N, workspace, status, epi, s));
}

}  // namespace

int gemm_entry(const void* x, const void* packed, const void* scales, int has_zeros, void* y,
               int B, int K, int N, int group_size, void* workspace, size_t ws_bytes, int path,
               void* stream) {
    return gemm_impl(x, packed, scales, has_zeros, y, B, K, N, group_size, workspace, ws_bytes,
                     path, stream);
}

#ifdef W4A16_DEBUG
static std::atomic<size_t> g_code_bound_cut{0};
#endif

size_t code_bound_bytes(int K, int N) {
    const size_t full = packed_code_bytes(K, N);
#ifdef W4A16_DEBUG
    const size_t cut = g_code_bound_cut.load(std::memory_order_relaxed);
    return cut < full ? full - cut : 0;
#else
    return full;
#endif
}

cudaError_t set_smem_limit(const void* kernel, size_t bytes) {
    static std::mutex mu;
    static std::unordered_map<const void*, size_t> set[64];  // per device: the limit set
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64)
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)bytes);
    std::lock_guard<std::mutex> lock(mu);
    auto it = set[dev].find(kernel);
    if (it != set[dev].end() && it->second >= bytes) return cudaSuccess;
    const cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err == cudaSuccess) set[dev][kernel] = bytes;
    return err;
}

cudaError_t launch_with_pdl(const void* func, dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, func, args);
}

}  // namespace w4a16

using namespace w4a16;

extern "C" {

size_t w4a16_packed_bytes(int K, int N, int group_size, int has_zeros) {
    if (group_size != kGroup || !shape_ok(K, N)) return 0;
    return packed_total_bytes(K, N, has_zeros != 0);
}

size_t w4a16_workspace_bytes(int B, int K, int N, int group_size) {
    if (group_size != kGroup || !shape_ok(K, N) || B < 1 || B > kMaxB) return (size_t)-1;
    // Enough for whichever path a call may take (auto or forced).
    size_t a = path_workspace(W4A16_PATH_SKINNY, B, K, N);
    if (tc_available()) {
        const size_t b = path_workspace(W4A16_PATH_TCGEN05, B, K, N);
        if (b > a) a = b;
    }
    return a;
}

w4a16_status w4a16_pack(const uint32_t* qweight, const uint32_t* qzeros, int K, int N,
                        int group_size, void* packed, void* stream) {
    if (group_size != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (!shape_ok(K, N)) return W4A16_ERR_SHAPE;
    if (!qweight || !packed) return W4A16_ERR_NULL;
    if (!aligned16(qweight) || !aligned16(packed) || (qzeros && !aligned16(qzeros)))
        return W4A16_ERR_ALIGN;
    return from_cuda(launch_repack(qweight, qzeros, K, N, packed, static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_gemm(const void* x, const void* packed, const void* scales, int has_zeros,
                        void* y, int B, int K, int N, int group_size, void* workspace,
                        size_t ws_bytes, void* stream) {
    return gemm_impl(x, packed, scales, has_zeros, y, B, K, N, group_size, workspace, ws_bytes,
                     W4A16_PATH_AUTO, stream);
}

w4a16_status w4a16_gemm_path(const void* x, const void* packed, const void* scales,
                             int has_zeros, void* y, int B, int K, int N, int group_size,
                             void* workspace, size_t ws_bytes, int path, void* stream) {
    return gemm_impl(x, packed, scales, has_zeros, y, B, K, N, group_size, workspace, ws_bytes,
                     path, stream);
}

w4a16_status w4a16_dequant_ref(const void* packed, const void* scales, int has_zeros, void* w,
                               int K, int N, int group_size, void* stream) {
    if (group_size != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (!shape_ok(K, N)) return W4A16_ERR_SHAPE;
    if (!packed || !scales || !w) return W4A16_ERR_NULL;
    if (!aligned16(packed) || !aligned16(scales) || !aligned16(w)) return W4A16_ERR_ALIGN;
    return from_cuda(launch_dequant_ref(packed, scales, has_zeros != 0, w, K, N, false,
                                        static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_dequant_ref_f16(const void* packed, const void* scales, int has_zeros, void* w,
                                   int K, int N, int group_size, void* stream) {
    if (group_size != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (!shape_ok(K, N)) return W4A16_ERR_SHAPE;
    if (!packed || !scales || !w) return W4A16_ERR_NULL;
    if (!aligned16(packed) || !aligned16(scales) || !aligned16(w)) return W4A16_ERR_ALIGN;
    return from_cuda(launch_dequant_ref(packed, scales, has_zeros != 0, w, K, N, true,
                                        static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_gemm_f16(const void* x, const void* packed, const void* scales, int has_zeros,
                            void* y, int B, int K, int N, int group_size, void* workspace,
                            size_t ws_bytes, void* stream) {
    Epilogue epi;
    epi.f16 = true;
    return gemm_impl(x, packed, scales, has_zeros, y, B, K, N, group_size, workspace, ws_bytes,
                     W4A16_PATH_AUTO, stream, 0, epi);
}

w4a16_status w4a16_gemm_f16_path(const void* x, const void* packed, const void* scales,
                                 int has_zeros, void* y, int B, int K, int N, int group_size,
                                 void* workspace, size_t ws_bytes, int path, void* stream) {
    Epilogue epi;
    epi.f16 = true;
    return gemm_impl(x, packed, scales, has_zeros, y, B, K, N, group_size, workspace, ws_bytes,
                     path, stream, 0, epi);
}

w4a16_status w4a16_gemm_fused(const void* x, const void* packed, const void* scales,
                              int has_zeros, const void* bias, int epilogue, void* y, int B, int K,
                              int N, int group_size, void* workspace, size_t ws_bytes,
                              void* stream) {
    if ((epilogue & ~(W4A16_EPI_BIAS | W4A16_EPI_SILU_MUL)) != 0) return W4A16_ERR_UNSUPPORTED;
    const bool want_bias = (epilogue & W4A16_EPI_BIAS) != 0;
    if (want_bias && bias == nullptr) return W4A16_ERR_NULL;
    if (want_bias && !aligned16(bias)) return W4A16_ERR_ALIGN;
    Epilogue epi;
    epi.bias = want_bias ? static_cast<const uint16_t*>(bias) : nullptr;
    epi.mode = epilogue;
    return gemm_impl(x, packed, scales, has_zeros, y, B, K, N, group_size, workspace, ws_bytes,
                     W4A16_PATH_AUTO, stream, 0, epi);
}

size_t w4a16_grouped_workspace_bytes(int T, int E, int max_rows, int K, int N, int group_size) {
    if (group_size != kGroup || !shape_ok(K, N) || T < 1 || T > kMaxB || E < 1 ||
        E > kMaxGroupedExperts || max_rows < 1)
        return (size_t)-1;
    return skinny_workspace_bytes(plan_skinny_grouped(T, E, max_rows, K, N, num_sms()), T, N);
}

w4a16_status w4a16_gemm_grouped(const void* x, const int* offsets, int E, int T,
                                const void* packed, const void* scales, int has_zeros, void* y,
                                int max_rows, int K, int N, int group_size, void* workspace,
                                size_t ws_bytes, void* stream) {
    if (group_size != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (!shape_ok(K, N) || T < 1 || T > kMaxB || E < 1 || E > kMaxGroupedExperts ||
        max_rows < 1)
        return W4A16_ERR_SHAPE;
    if (!x || !offsets || !packed || !scales || !y || !workspace) return W4A16_ERR_NULL;
    if (!aligned16(x) || !aligned16(packed) || !aligned16(scales) || !aligned16(y) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(offsets) & 3u) != 0)
        return W4A16_ERR_ALIGN;
    const SkinnyPlan p = plan_skinny_grouped(T, E, max_rows, K, N, num_sms());
    if (ws_bytes < skinny_workspace_bytes(p, T, N)) return W4A16_ERR_WORKSPACE;
    unsigned int* status = device_status_word();
    if (status == nullptr) return W4A16_ERR_CUDA;
    return from_cuda(launch_skinny_grouped(p, x, offsets, E, packed, scales, has_zeros != 0, y, T,
                                           K, N, workspace, status,
                                           static_cast<cudaStream_t>(stream)));
}

w4a16_status w8a8_fp8_quantize_act(const void* x, int B, int K, void* xq, float* sx,
                                   void* stream) {
    if (!shape_ok(K, 8) || B < 1 || B > kMaxB) return W4A16_ERR_SHAPE;
    if (!x || !xq || !sx) return W4A16_ERR_NULL;
    if (!aligned16(x) || !aligned16(xq) || (reinterpret_cast<uintptr_t>(sx) & 3u) != 0)
        return W4A16_ERR_ALIGN;
    return from_cuda(launch_fp8_quantize_rows(x, B, K, xq, sx, static_cast<cudaStream_t>(stream)));
}

w4a16_status w8a8_fp8_quantize_weight(const void* w, int K, int N, void* wq, float* sw,
                                      void* stream) {
    if (!shape_ok(K, N)) return W4A16_ERR_SHAPE;
    if (!w || !wq || !sw) return W4A16_ERR_NULL;
    if (!aligned16(w) || !aligned16(wq) || (reinterpret_cast<uintptr_t>(sw) & 3u) != 0)
        return W4A16_ERR_ALIGN;
    return from_cuda(launch_fp8_quantize_cols(w, K, N, wq, sw, static_cast<cudaStream_t>(stream)));
}

size_t w8a8_fp8_packed_bytes(int K, int N) {
    return shape_ok(K, N) ? fp8_packed_bytes(K, N) : 0;
}

w4a16_status w8a8_fp8_pack_weight(const void* wq, int K, int N, void* packed, void* stream) {
    if (!shape_ok(K, N)) return W4A16_ERR_SHAPE;
    if (!wq || !packed) return W4A16_ERR_NULL;
    if (!aligned16(wq) || !aligned16(packed)) return W4A16_ERR_ALIGN;
    return from_cuda(launch_fp8_pack(wq, K, N, packed, static_cast<cudaStream_t>(stream)));
}

size_t w8a8_fp8_workspace_bytes(int B, int K, int N) {
    if (!shape_ok(K, N) || B < 1 || B > kMaxB) return (size_t)-1;
    return fp8_workspace_bytes(plan_fp8(B, K, N, num_sms()), B, N);
}

w4a16_status w8a8_fp8_gemm(const void* xq, const float* sx, const void* packed, const float* sw,
                           void* y, int B, int K, int N, void* workspace, size_t ws_bytes,
                           void* stream) {
    if (!shape_ok(K, N) || B < 1 || B > kMaxB) return W4A16_ERR_SHAPE;
    if (!xq || !sx || !packed || !sw || !y) return W4A16_ERR_NULL;
    if (!aligned16(xq) || !aligned16(packed) || !aligned16(y) ||
        ((reinterpret_cast<uintptr_t>(sx) | reinterpret_cast<uintptr_t>(sw)) & 3u) != 0)
        return W4A16_ERR_ALIGN;
    const Fp8Plan p = plan_fp8(B, K, N, num_sms());
    const size_t need = fp8_workspace_bytes(p, B, N);
    if (need > 0) {
        if (workspace == nullptr) return W4A16_ERR_NULL;
        if (!aligned16(workspace)) return W4A16_ERR_ALIGN;
        if (ws_bytes < need) return W4A16_ERR_WORKSPACE;
    }
    if (!tc_available()) return W4A16_ERR_UNSUPPORTED;
    unsigned int* status = device_status_word();
    if (status == nullptr) return W4A16_ERR_CUDA;
    return from_cuda(launch_fp8_gemm(p, xq, sx, packed, sw, y, B, K, N, workspace, status,
                                     static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_quantize_rtn(const void* w, int K, int N, int group_size, uint32_t* qweight,
                                void* scales, void* stream) {
    if (group_size != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (!shape_ok(K, N)) return W4A16_ERR_SHAPE;
    if (!w || !qweight || !scales) return W4A16_ERR_NULL;
    if (!aligned16(w) || !aligned16(qweight) || !aligned16(scales)) return W4A16_ERR_ALIGN;
    return from_cuda(launch_quantize(w, K, N, qweight, scales, static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_debug_forced_timeout(const void* x, const void* packed, const void* scales,
                                        int has_zeros, void* y, int B, int K, int N,
                                        int group_size, void* workspace, size_t ws_bytes,
                                        int wait_ms, void* stream) {
    if (wait_ms < 1 || wait_ms > 10000) return W4A16_ERR_UNSUPPORTED;
    return gemm_impl(x, packed, scales, has_zeros, y, B, K, N, group_size, workspace, ws_bytes,
                     W4A16_PATH_TCGEN05, stream, wait_ms);
}

int w4a16_select_path(int B, int K, int N) {
    if (!shape_ok(K, N) || B < 1 || B > kMaxB) return -1;
    return choose_path(B, K, N);
}

w4a16_status w4a16_describe_plan(int B, int K, int N, int group_size, int num_sms_arg,
                                 w4a16_plan_info* out) {
    if (out == nullptr) return W4A16_ERR_NULL;
    *out = w4a16_plan_info{};
    if (group_size != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (!shape_ok(K, N) || B < 1 || B > kMaxB || num_sms_arg < 0) return W4A16_ERR_SHAPE;
    int sms = num_sms_arg;
    int path;
    if (sms == 0) {  // the current device
        if (device_info().sms <= 0) return W4A16_ERR_CUDA;
        sms = num_sms();
        path = choose_path(B, K, N);
    } else {  // a GB300-class device with that many SMs
        const int forced = forced_path();
        path = forced == W4A16_PATH_SKINNY ? W4A16_PATH_SKINNY
               : forced == W4A16_PATH_TCGEN05 ? W4A16_PATH_TCGEN05
               : (B <= kSkinnyMaxB ? W4A16_PATH_SKINNY : W4A16_PATH_TCGEN05);
    }
    if (path == W4A16_PATH_SKINNY) {
        const SkinnyPlan p = num_sms_arg == 0 ? skinny_plan(B, K, N) : plan_skinny(B, K, N, sms);
        const PlanResources r = skinny_resources(p);
        out->kernel = 0;
        out->batch_rows = 8 * p.nt;
        out->batch_tiles = p.batch_chunks;
        out->col_tiles = p.col_blocks;
        out->k_splits = p.split;
        out->groups_per_split = p.gps;
        out->grid = p.grid;
        out->ctas_per_sm = r.ctas_per_sm;
        out->code_slots = r.code_slots;
        out->block_rows = r.block_rows;
        out->smem_bytes = r.smem;
        out->workspace_bytes = skinny_workspace_bytes(p, B, N);
        return W4A16_OK;
    }
    const TcPlan p = num_sms_arg == 0 ? tc_plan(B, K, N) : plan_tc(B, K, N, sms);
    out->batch_rows = p.bn;
    out->batch_tiles = p.batch_tiles;
    out->col_tiles = p.col_tiles;
    out->k_splits = p.split;
    out->groups_per_split = p.kb_per_split / 2;
    out->grid = p.grid;
    out->ctas_per_sm = 1;
    out->workspace_bytes = tc_workspace_bytes(p, B, N);
    if (!p.wide) {  // the multi-issuer TMEM kernel (forced path at <= 16 rows)
        out->kernel = 1;
        out->issuers = p.issuers;
        out->acc_buffers = p.bufs;
        out->tile_slots = p.a_slots;
        out->block_rows = 64;
        return W4A16_OK;
    }
    const PlanResources r = wide_resources(p, B, N);
    out->kernel = 2;
    out->issuers = r.issuers;
    out->acc_buffers = r.acc_bufs;
    out->tile_slots = r.tile_slots;
    out->x_slots = r.x_slots;
    out->code_slots = r.code_slots;
    out->block_rows = r.block_rows;
    out->tmem_cols = r.tmem_cols;
    out->smem_bytes = r.smem;
    return W4A16_OK;
}

const char* w4a16_kernel_name(int B, int K, int N) {
    if (!shape_ok(K, N) || B < 1 || B > kMaxB) return "invalid";
    if (choose_path(B, K, N) == W4A16_PATH_SKINNY) return "skinny_kernel";
    return tc_plan(B, K, N).wide ? "wide_kernel" : "tc_kernel";
}

w4a16_status w4a16_device_status(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return W4A16_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return W4A16_ERR_CUDA;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess)
            return W4A16_ERR_CUDA;
    }
    if (v == 0) return W4A16_OK;
    if (v == kStatusBadBlob) return W4A16_ERR_UNSUPPORTED;
    return v == kStatusBounds ? W4A16_ERR_BOUNDS : W4A16_ERR_TIMEOUT;
}

int w4a16_debug_build(void) {
#ifdef W4A16_DEBUG
    return 1;
#else
    return 0;
#endif
}

w4a16_status w4a16_debug_shrink_code_bound(size_t bytes) {
#ifdef W4A16_DEBUG
    g_code_bound_cut.store(bytes, std::memory_order_relaxed);
    return W4A16_OK;
#else
    (void)bytes;
    return W4A16_ERR_UNSUPPORTED;
#endif
}

w4a16_status w4a16_packed_check(const void* packed, int K, int N, int group_size, int has_zeros,
                                void* stream) {
    if (group_size != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (!shape_ok(K, N)) return W4A16_ERR_SHAPE;
    if (packed == nullptr) return W4A16_ERR_NULL;
    if (!aligned16(packed)) return W4A16_ERR_ALIGN;
    uint32_t got[4] = {0, 0, 0, 0};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const char* tag = static_cast<const char*>(packed) + packed_tag_offset(K, N, has_zeros != 0);
    if (cudaMemcpyAsync(got, tag, sizeof got, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return W4A16_ERR_CUDA;
    const BlobTag want = blob_tag(K, N, has_zeros != 0);
    if (got[0] != want.w[0] || got[1] != want.w[1]) return W4A16_ERR_UNSUPPORTED;
    if (got[2] != want.w[2] || got[3] != want.w[3]) return W4A16_ERR_SHAPE;
    return W4A16_OK;
}

const char* w4a16_status_string(w4a16_status status) {
    switch (status) {
        case W4A16_OK: return "ok";
        case W4A16_ERR_NULL: return "a required pointer is NULL";
        case W4A16_ERR_SHAPE: return "invalid shape (need B >= 1, K % 128 == 0, N % 8 == 0)";
        case W4A16_ERR_ALIGN: return "pointer not 16-byte aligned";
        case W4A16_ERR_UNSUPPORTED: return "unsupported group size or kernel path";
        case W4A16_ERR_WORKSPACE: return "workspace too small";
        case W4A16_ERR_CUDA: return "CUDA error";
        case W4A16_ERR_TIMEOUT: return "device-side wait timed out";
        case W4A16_ERR_BOUNDS: return "device-side bounds check failed (debug build)";
    }
    return "unknown status";
}

}  // extern "C"
