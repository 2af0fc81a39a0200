// gemm_cfg_single16.cu -- kernels of the single16 tile configuration (all output
// types), in a translation unit of their own so configurations compile in parallel.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND(single16, CfgSingle16, kCfgSingle16)
}  // namespace tcdt_host
