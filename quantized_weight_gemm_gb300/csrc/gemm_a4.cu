// Instantiations of the tensor-core GEMM for MXFP4 weights x MXFP4 activations (W4A4,
// kind::mxf4 block-scaled MMAs on operands read from shared memory).
#include "gemm_kernel.cuh"

namespace qgemm {
cudaError_t launch_gemm_a4(const GemmPlan& plan, const CUtensorMap& tmap, const GemmArgs& args,
                           cudaStream_t st) {
  return launch_gemm_impl<false, DM_W4A4>(plan, tmap, args, st);
}
}  // namespace qgemm
