// Instantiations of the tensor-core GEMM for BF16 activations (kind::f16), decode mode NVFP4.
#include "gemm_kernel.cuh"

namespace qgemm {
cudaError_t launch_gemm_a16_nvfp4(const GemmPlan& plan, const CUtensorMap& tmap,
                                  const GemmArgs& args, cudaStream_t st) {
  return launch_gemm_impl<false, DM_NVFP4>(plan, tmap, args, st);
}
}  // namespace qgemm
