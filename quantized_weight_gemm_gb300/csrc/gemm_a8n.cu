// Instantiations of the tensor-core GEMM for MXFP4 weights x FP8 activations with the e2m1
// codes as the MMA's FP4 operand (kind::mxf8f6f4 block-scaled, A and B from shared memory).
#include "gemm_kernel.cuh"

namespace qgemm {
cudaError_t launch_gemm_a8n(const GemmPlan& plan, const CUtensorMap& tmap, const GemmArgs& args,
                            cudaStream_t st) {
  return launch_gemm_impl<true, DM_W4A8N>(plan, tmap, args, st);
}
}  // namespace qgemm
