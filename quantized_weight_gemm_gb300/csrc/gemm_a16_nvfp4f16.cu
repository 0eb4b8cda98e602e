// Instantiations of the tensor-core GEMM for BF16 activations converted to FP16 (kind::f16
// on FP16 operands), decode mode NVFP4 through the hardware e2m1x2 and e4m3x2 conversions
// (narrow token tiles).
#include "gemm_kernel.cuh"

namespace qgemm {
cudaError_t launch_gemm_a16_nvfp4f16(const GemmPlan& plan, const CUtensorMap& tmap,
                                      const GemmArgs& args, cudaStream_t st) {
  return launch_gemm_impl<false, DM_NVFP4_F16>(plan, tmap, args, st);
}
}  // namespace qgemm
