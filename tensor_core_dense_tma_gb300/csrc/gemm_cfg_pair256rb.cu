// gemm_cfg_pair256rb.cu -- the pair256 tile configuration with the row-bulk
// epilogue (fp32 output only), in a translation unit of its own.
#include "gemm_internal.cuh"

namespace tcdt_host {
gemm_status_t prepare_pair256rb(gemm_plan* plan, int slot) {
    if (slot != 0) return GEMM_ERR_UNSUPPORTED;
    return prepare<CfgPair256Rb>(plan, kCfgPair256Rb, 0);
}

gemm_status_t launch_pair256rb(gemm_plan* plan, int slot, const Choice& ch, const Problem& pr, const void* C,
                               void* D, int64_t ldc, float alpha, float beta, cudaStream_t s) {
    const gemm_status_t st = prepare_pair256rb(plan, slot);
    if (st != GEMM_OK) return st;
    return launch_tc<CfgPair256Rb>(plan, ch, pr, C, D, ldc, alpha, beta, GEMM_F32, s);
}
}  // namespace tcdt_host
