// Instantiations of the tensor-core GEMM for FP8 activations (kind::mxf8f6f4 block-scaled).
#include "gemm_kernel.cuh"

namespace qgemm {
cudaError_t launch_gemm_a8(const GemmPlan& plan, const CUtensorMap& tmap, const GemmArgs& args,
                           cudaStream_t st) {
  return launch_gemm_impl<true>(plan, tmap, args, st);
}
int gemm_smem_bytes_a8(int bnt) { return smem_bytes_impl<true>(bnt); }

cudaError_t launch_gemm_a16(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
int gemm_smem_bytes_a16(int bnt);

cudaError_t launch_gemm(bool fp8, const GemmPlan& plan, const CUtensorMap& tmap,
                        const GemmArgs& args, cudaStream_t st) {
  return fp8 ? launch_gemm_a8(plan, tmap, args, st) : launch_gemm_a16(plan, tmap, args, st);
}
int gemm_smem_bytes(bool fp8, int bnt) {
  return fp8 ? gemm_smem_bytes_a8(bnt) : gemm_smem_bytes_a16(bnt);
}
}  // namespace qgemm
