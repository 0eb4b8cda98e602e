// Instantiations of the tensor-core GEMM for BF16 activations (kind::f16).
#include "gemm_kernel.cuh"

namespace qgemm {
cudaError_t launch_gemm_a16(const GemmPlan& plan, const CUtensorMap& tmap, const GemmArgs& args,
                            cudaStream_t st) {
  return launch_gemm_impl<false>(plan, tmap, args, st);
}
int gemm_smem_bytes_a16(int bnt) { return smem_bytes_impl<false>(bnt); }
}  // namespace qgemm
