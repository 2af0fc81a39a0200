// gemm_cfg_pair256_ep.cu -- kernels of the pair256 tile configuration with the fused
// epilogue (bias, scales, activation), in a translation unit of their own.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_EP(pair256, CfgPair256)
}  // namespace tcdt_host
