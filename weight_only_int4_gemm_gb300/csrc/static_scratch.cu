// static_scratch.cu -- w4a16_gemm for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc at all: code running
// where allocation is forbidden or unavailable (for example inside a region
// whose memory was planned up front, or a host environment that owns every
// device allocation itself) still needs the split-K GEMM, whose kernels keep
// partial sums and arrival counters in scratch memory.  This file gives them
// one entry point whose scratch is a file-scope device array compiled into
// the library, so the call itself allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = (size_t)4 << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the array on the current device, looked up once per
// device (with that device current) on the first call there.
void* static_scratch_address(int* err) {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *err = W4A16_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
            *err = W4A16_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace
}  // namespace w4a16

extern "C" w4a16_status w4a16_gemm_static_scratch(const void* x, const void* packed,
                                                  const void* scales, int has_zeros, void* y,
                                                  int B, int K, int N, int group_size,
                                                  void* stream) {
    using namespace w4a16;
    // The same bound a caller gets from w4a16_workspace_bytes (enough for any
    // path), so the refusal below is exactly the documented one.
    const size_t need = w4a16_workspace_bytes(B, K, N, group_size);
    if (need == (size_t)-1) {
        // let the common validation report the precise problem
        return static_cast<w4a16_status>(gemm_entry(x, packed, scales, has_zeros, y, B, K, N,
                                                    group_size, nullptr, 0, W4A16_PATH_AUTO,
                                                    stream));
    }
    if (need > kStaticScratchBytes) return W4A16_ERR_WORKSPACE;
    int err = W4A16_OK;
    void* scratch = static_scratch_address(&err);
    if (scratch == nullptr) return static_cast<w4a16_status>(err);
    // The array keeps whatever the previous call left.  The kernels expect
    // all of the scratch they use at zero: the arrival counters and scheduler
    // words, and the fp32 accumulator the split-K partial sums are added
    // into (red.global.add reads it).  A normal call leaves it at zero, but a
    // call whose bounded wait expired (W4A16_ERR_TIMEOUT) can leave partial
    // sums and counts behind, and the caller cannot reach this array to
    // repair it -- so every call clears all `need` bytes first (at most the
    // array's size; one memset on the caller's stream, no allocation).
    if (need > 0 && cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) !=
                        cudaSuccess)
        return W4A16_ERR_CUDA;
    return static_cast<w4a16_status>(gemm_entry(x, packed, scales, has_zeros, y, B, K, N,
                                                group_size, scratch, kStaticScratchBytes,
                                                W4A16_PATH_AUTO, stream));
}
