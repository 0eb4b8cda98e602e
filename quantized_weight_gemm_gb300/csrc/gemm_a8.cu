// Instantiations of the tensor-core GEMM for FP8 activations (kind::mxf8f6f4 block-scaled),
// and the dispatch over activation format and decode mode.
#include "gemm_kernel.cuh"

namespace qgemm {
cudaError_t launch_gemm_a16_zp_g1(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_a16_sym_g1(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_a16_any(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_a16_mxfp4(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_a16_mxint4(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_a16_nvfp4(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_a4(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_a8n(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_a16_mxfp4f16(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);
cudaError_t launch_gemm_a16_nvfp4f16(const GemmPlan&, const CUtensorMap&, const GemmArgs&, cudaStream_t);

cudaError_t launch_gemm(bool fp8, const GemmPlan& plan, const CUtensorMap& tmap,
                        const GemmArgs& args, cudaStream_t st) {
  if (fp8)
    return decode_mode(args.L) == DM_W4A8N ? launch_gemm_a8n(plan, tmap, args, st)
                                           : launch_gemm_impl<true, DM_MXFP4>(plan, tmap, args, st);
  switch (decode_mode(args.L)) {
    case DM_INT4_ZP_G1: return launch_gemm_a16_zp_g1(plan, tmap, args, st);
    case DM_INT4_SYM_G1: return launch_gemm_a16_sym_g1(plan, tmap, args, st);
    case DM_MXFP4:
      return plan.mx_f16 ? launch_gemm_a16_mxfp4f16(plan, tmap, args, st)
                         : launch_gemm_a16_mxfp4(plan, tmap, args, st);
    case DM_MXINT4: return launch_gemm_a16_mxint4(plan, tmap, args, st);
    case DM_NVFP4:
      return plan.mx_f16 ? launch_gemm_a16_nvfp4f16(plan, tmap, args, st)
                         : launch_gemm_a16_nvfp4(plan, tmap, args, st);
    case DM_W4A4: return launch_gemm_a4(plan, tmap, args, st);
    default: return launch_gemm_a16_any(plan, tmap, args, st);
  }
}

int gemm_smem_bytes(bool fp8, int bnt) {
  return fp8 ? smem_bytes_impl<true>(bnt) : smem_bytes_impl<false>(bnt);
}
int gemm_x_box_slabs(bool fp8, int bnt) {
  return fp8 ? x_box_slabs_impl<true>(bnt) : x_box_slabs_impl<false>(bnt);
}
}  // namespace qgemm
