// gemm_cfg_single64_f8.cu -- kernels of the single64 tile configuration for 8-bit (E4M3 / E5M2) operands,
// tcgen05.mma kind::f8f6f4 (fp32 accumulation, all output
// types), in a translation unit of their own so configurations compile in parallel.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_IN(single64, CfgSingle64, f8, tcdt::kInF8)
}  // namespace tcdt_host
