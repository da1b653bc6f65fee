// gemm_instances.cuh -- the four GEMM kernels of the path for one element
// size, and their launchers.  Included once per element type so the two
// instantiations compile in parallel.
#pragma once
#include "epilogues.cuh"
#include "launch.h"

namespace flce {

// bf16: CTA pairs (cta_group::2, 256 x 256 tiles); dW = G^T X reads both
// operands MN-major, dX = G W reads W MN-major.
// fp32 (tf32 products): single CTAs, every operand K-major; the path hands
// the gradient GEMMs transposed copies (tf32 MMAs here take K-major operands
// only).
template <int ELT>
struct Kernels {
  using GradEpi = EpiGradLogits<ELT>;
  static constexpr bool kPair = (ELT == 2);
  static constexpr bool kMN = (ELT == 2);
  static constexpr auto lse = gemm_kernel<ELT, false, false, kPair, EpiRowLse>;
  static constexpr auto grad = gemm_kernel<ELT, false, false, kPair, GradEpi>;
  static constexpr auto dw = gemm_kernel<ELT, kMN, kMN, kPair, EpiStoreF32>;
  static constexpr auto dx = gemm_kernel<ELT, false, kMN, kPair, EpiStoreF32>;

  template <class KernelT>
  static cudaError_t set_smem(KernelT k) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GEMM_SMEM_BYTES);
  }

  // Shared-memory limits; *max_units = scheduling units (CTAs or CTA pairs)
  // that can be resident at once.
  static cudaError_t prepare(int sms, int* max_units) {
    cudaError_t e;
    if ((e = set_smem(lse)) != cudaSuccess) return e;
    if ((e = set_smem(grad)) != cudaSuccess) return e;
    if ((e = set_smem(dw)) != cudaSuccess) return e;
    if ((e = set_smem(dx)) != cudaSuccess) return e;
    if (!kPair) {
      *max_units = sms;
      return cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    fill_config(&cfg, attr, sms, nullptr);
    int clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&clusters, lse, &cfg)) != cudaSuccess) return e;
    *max_units = clusters > 0 ? clusters : 1;
    return cudaSuccess;
  }

  static void fill_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int units,
                          cudaStream_t s) {
    cfg->gridDim = dim3(static_cast<unsigned>(units * (kPair ? 2 : 1)));
    cfg->blockDim = dim3(NUM_THREADS);
    cfg->dynamicSmemBytes = GEMM_SMEM_BYTES;
    cfg->stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the kernel's prologue overlaps the tail
    // of the previous kernel in the stream (the kernel waits on its
    // predecessor with griddepcontrol.wait before touching global memory)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 2;
  }

  template <class KernelT, class P>
  static cudaError_t launch(KernelT k, const CUtensorMap& A, const CUtensorMap& B,
                            const CUtensorMap& out, const GemmGrid& g, const P& p, int units,
                            cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    fill_config(&cfg, attr, units, s);
    return cudaLaunchKernelEx(&cfg, k, A, B, out, g, p);
  }

  static cudaError_t run_lse(const CUtensorMap& A, const CUtensorMap& B, const GemmGrid& g,
                             const RowLseParams& p, int units, cudaStream_t s) {
    EpiRowLse::Params ep{p.target, p.partial, p.st, p.N, p.V, p.vtile_off};
    return launch(lse, A, B, A, g, ep, units, s);
  }

  static cudaError_t run_grad(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                              const GemmGrid& g, const GradLogitsParams& p, int units,
                              cudaStream_t s) {
    typename GradEpi::Params ep{p.target, p.lse2, p.scalars, p.N, p.V, p.ignore_index,
                                p.vocab_off};
    return launch(grad, A, B, out, g, ep, units, s);
  }

  static cudaError_t run_dw(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                            const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s) {
    EpiStoreF32::Params ep{p.x_off, p.y_off, p.reduce};
    return launch(dw, A, B, out, g, ep, units, s);
  }

  static cudaError_t run_dx(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                            const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s) {
    EpiStoreF32::Params ep{p.x_off, p.y_off, p.reduce};
    return launch(dx, A, B, out, g, ep, units, s);
  }
};

}  // namespace flce
