// Prefill path of the expert FFN (tcgen05 block-scaled grouped GEMM).
#include "internal.h"

namespace moe {

size_t prefill_workspace_bytes(int T, int k, int H, int I) {
    (void)T; (void)k; (void)H; (void)I;
    return 0;
}

int launch_prefill_ffn(const FfnArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    (void)a; (void)ws; (void)ws_bytes; (void)s;
    return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
