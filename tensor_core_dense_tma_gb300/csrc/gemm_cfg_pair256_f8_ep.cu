// gemm_cfg_pair256_f8_ep.cu -- kernels of the pair256 tile configuration for 8-bit (E4M3 / E5M2) operands
// with the fused epilogue (bias, scales, activation), in a translation unit of their own.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_IN_EP(pair256, CfgPair256, f8, tcdt::kInF8)
}  // namespace tcdt_host
