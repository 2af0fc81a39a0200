// gemm_cfg_pair256.cu -- kernels of the pair256 tile configuration (all output
// types), in a translation unit of their own so configurations compile in parallel.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND(pair256, CfgPair256, kCfgPair256)
}  // namespace tcdt_host
