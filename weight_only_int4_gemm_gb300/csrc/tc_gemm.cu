// tc_gemm.cu -- tcgen05/TMEM tensor-core W4A16 GEMM (large batch).
#include "launch.cuh"

namespace w4a16 {

bool tc_available() { return false; }

TcPlan plan_tc(int B, int K, int N, int num_sms) {
    (void)K;
    (void)num_sms;
    TcPlan p{};
    p.bn = 256;
    p.batch_tiles = (B + 255) / 256;
    p.col_tiles = (N + 127) / 128;
    p.kb_per_split = 0;
    p.split = 1;
    return p;
}

size_t tc_workspace_bytes(const TcPlan&, int, int) { return 0; }

cudaError_t launch_tc(const TcPlan&, const void*, const void*, const void*, bool, void*, int, int,
                      int, void*, unsigned int*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace w4a16
