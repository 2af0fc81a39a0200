// gemm_cfg_single64_ep.cu -- kernels of the single64 tile configuration with the fused
// epilogue (bias, scales, activation), in a translation unit of their own.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_EP(single64, CfgSingle64)
}  // namespace tcdt_host
