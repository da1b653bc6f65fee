// gemm_bf16.cu -- bf16 instantiations of the path's GEMM kernels.
#include "gemm_instances.cuh"

namespace flce {
using K = Kernels<2>;
cudaError_t gemm_prepare_bf16(int sms, int* max_units) { return K::prepare(sms, max_units); }
cudaError_t launch_logits_lse_bf16(const CUtensorMap& A, const CUtensorMap& B, const GemmGrid& g,
                                   const RowLseParams& p, int units, cudaStream_t s) {
  return K::run_lse(A, B, g, p, units, s);
}
cudaError_t launch_logits_grad_bf16(const CUtensorMap& A, const CUtensorMap& B,
                                    const CUtensorMap& out, const GemmGrid& g,
                                    const GradLogitsParams& p, int units, cudaStream_t s) {
  return K::run_grad(A, B, out, g, p, units, s);
}
cudaError_t launch_dw_bf16(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                           const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s) {
  return K::run_dw(A, B, out, g, p, units, s);
}
cudaError_t launch_dx_bf16(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                           const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s) {
  return K::run_dx(A, B, out, g, p, units, s);
}
}  // namespace flce
