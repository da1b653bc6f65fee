// gemm_instances.cuh -- the four GEMM kernels of the path for one element
// size, and their launchers.  Included once per element type so the two
// instantiations compile in parallel.
#pragma once
#include "epilogues.cuh"
#include "launch.h"

namespace flce {

// bf16: dW = G^T X reads both operands MN-major, dX = G W reads W MN-major.
// fp32 (tf32 products): every operand is K-major; the path hands these GEMMs
// transposed copies instead (tf32 MMAs here take K-major operands only).
template <int ELT>
struct Kernels {
  using GradEpi = EpiGradLogits<ELT>;
  static constexpr bool kMN = (ELT == 2);
  static constexpr auto lse = gemm_kernel<ELT, false, false, EpiRowLse>;
  static constexpr auto grad = gemm_kernel<ELT, false, false, GradEpi>;
  static constexpr auto dw = gemm_kernel<ELT, kMN, kMN, EpiStoreF32>;
  static constexpr auto dx = gemm_kernel<ELT, false, kMN, EpiStoreF32>;

  static cudaError_t prepare() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(lse, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  GEMM_SMEM_BYTES)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(grad, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  GEMM_SMEM_BYTES)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(dw, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  GEMM_SMEM_BYTES)) != cudaSuccess)
      return e;
    return cudaFuncSetAttribute(dx, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GEMM_SMEM_BYTES);
  }

  static cudaError_t run_lse(const CUtensorMap& A, const CUtensorMap& B, const GemmGrid& g,
                             const RowLseParams& p, int grid, cudaStream_t s) {
    EpiRowLse::Params ep{p.target, p.partial, p.st, p.N, p.V};
    lse<<<grid, NUM_THREADS, GEMM_SMEM_BYTES, s>>>(A, B, A, g, ep);
    return cudaGetLastError();
  }

  static cudaError_t run_grad(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                              const GemmGrid& g, const GradLogitsParams& p, int grid,
                              cudaStream_t s) {
    typename GradEpi::Params ep{p.target, p.lse2, p.scalars, p.N, p.V, p.ignore_index,
                                p.vocab_off};
    grad<<<grid, NUM_THREADS, GEMM_SMEM_BYTES, s>>>(A, B, out, g, ep);
    return cudaGetLastError();
  }

  static cudaError_t run_dw(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                            const GemmGrid& g, const StoreParams& p, int grid, cudaStream_t s) {
    EpiStoreF32::Params ep{p.x_off, p.y_off, p.reduce};
    dw<<<grid, NUM_THREADS, GEMM_SMEM_BYTES, s>>>(A, B, out, g, ep);
    return cudaGetLastError();
  }

  static cudaError_t run_dx(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                            const GemmGrid& g, const StoreParams& p, int grid, cudaStream_t s) {
    EpiStoreF32::Params ep{p.x_off, p.y_off, p.reduce};
    dx<<<grid, NUM_THREADS, GEMM_SMEM_BYTES, s>>>(A, B, out, g, ep);
    return cudaGetLastError();
  }
};

}  // namespace flce
