// gemm_fp32.cu -- fp32 (tf32 tensor-core) instantiations of the path's GEMM kernels.
#include "gemm_instances.cuh"

namespace flce {
using K = Kernels<4>;
cudaError_t gemm_prepare_fp32(int sms, int* max_units) { return K::prepare(sms, max_units); }
cudaError_t launch_logits_lse_fp32(const CUtensorMap& A, const CUtensorMap& B, const GemmGrid& g,
                                   const RowLseParams& p, int units, cudaStream_t s) {
  return K::run_lse(A, B, g, p, units, s);
}
cudaError_t launch_logits_grad_fp32(const CUtensorMap& A, const CUtensorMap& B,
                                    const CUtensorMap& out, const GemmGrid& g,
                                    const GradLogitsParams& p, int units, cudaStream_t s) {
  return K::run_grad(A, B, out, g, p, units, s);
}
cudaError_t launch_dw_fp32(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                           const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s) {
  return K::run_dw(A, B, out, g, p, units, s);
}
cudaError_t launch_dx_fp32(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                           const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s) {
  return K::run_dx(A, B, out, g, p, units, s);
}
}  // namespace flce
