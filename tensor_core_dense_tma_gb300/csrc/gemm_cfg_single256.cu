// gemm_cfg_single256.cu -- kernels of the single256 tile configuration (all output
// types), in a translation unit of their own so configurations compile in parallel.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND(single256, CfgSingle256, kCfgSingle256)
}  // namespace tcdt_host
