// gemm_cfg_pair256_f8.cu -- kernels of the pair256 tile configuration for 8-bit (E4M3 / E5M2) operands,
// tcgen05.mma kind::f8f6f4 (fp32 accumulation, all output
// types), in a translation unit of their own so configurations compile in parallel.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_IN(pair256, CfgPair256, f8, tcdt::kInF8)
}  // namespace tcdt_host
