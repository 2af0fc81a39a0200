// gemm_cfg_single64_tf32.cu -- kernels of the single64 tile configuration for tf32 operands,
// tcgen05.mma kind::tf32 (fp32 accumulation, all output
// types), in a translation unit of their own so configurations compile in parallel.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_IN(single64, CfgSingle64, tf32, tcdt::kInTF32)
}  // namespace tcdt_host
