// gemm_cfg_pair224.cu -- kernels of the pair224 tile configuration (all output
// types), in a translation unit of their own so configurations compile in parallel.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND(pair224, CfgPair224, kCfgPair224)
}  // namespace tcdt_host
