// gemm_cfg_single16_tf32_ep.cu -- kernels of the single16 tile configuration for tf32 operands
// with the fused epilogue (bias, scales, activation), in a translation unit of their own.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_IN_EP(single16, CfgSingle16, tf32, tcdt::kInTF32)
}  // namespace tcdt_host
