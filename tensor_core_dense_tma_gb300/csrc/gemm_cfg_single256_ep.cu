// gemm_cfg_single256_ep.cu -- kernels of the single256 tile configuration with the fused
// epilogue (bias, scales, activation), in a translation unit of their own.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_EP(single256, CfgSingle256)
}  // namespace tcdt_host
