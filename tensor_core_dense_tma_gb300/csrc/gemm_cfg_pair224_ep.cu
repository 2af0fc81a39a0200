// gemm_cfg_pair224_ep.cu -- kernels of the pair224 tile configuration with the fused
// epilogue (bias, scales, activation), in a translation unit of their own.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_EP(pair224, CfgPair224)
}  // namespace tcdt_host
