// gemm_cfg_single16_ep.cu -- kernels of the single16 tile configuration with the fused
// epilogue (bias, scales, activation), in a translation unit of their own.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_EP(single16, CfgSingle16)
}  // namespace tcdt_host
