// gemm_cfg_single64.cu -- kernels of the single64 tile configuration (all output
// types), in a translation unit of their own so configurations compile in parallel.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND(single64, CfgSingle64, kCfgSingle64)
}  // namespace tcdt_host
