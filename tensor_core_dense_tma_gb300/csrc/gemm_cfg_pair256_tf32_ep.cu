// gemm_cfg_pair256_tf32_ep.cu -- kernels of the pair256 tile configuration for tf32 operands
// with the fused epilogue (bias, scales, activation), in a translation unit of their own.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_IN_EP(pair256, CfgPair256, tf32, tcdt::kInTF32)
}  // namespace tcdt_host
