// gemm_cfg_single16_tf32.cu -- kernels of the single16 tile configuration for tf32 operands,
// tcgen05.mma kind::tf32 (fp32 accumulation, all output
// types), in a translation unit of their own so configurations compile in parallel.
#include "gemm_internal.cuh"

namespace tcdt_host {
TCDT_DEFINE_KIND_IN(single16, CfgSingle16, tf32, tcdt::kInTF32)
}  // namespace tcdt_host
