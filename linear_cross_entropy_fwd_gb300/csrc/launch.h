// launch.h -- host-side launchers of the libflce kernels (internal).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "flce_internal.h"

namespace flce {

struct RowLseParams {
  Targets target;
  float* partial;
  float* st;
  int64_t N;
  int64_t V;
  int32_t vtile_off;  // vocabulary tile of the launch's first tile column
};

struct GradLogitsParams {
  Targets target;
  const float* lse2;
  const Scalars* scalars;
  int64_t N;
  int64_t V;
  int64_t ignore_index;
  int64_t vocab_off;
};

struct StoreParams {
  int32_t x_off;
  int32_t y_off;
  int32_t reduce;
};

// Set the dynamic shared-memory limit of every GEMM kernel on the current
// device; *max_units = scheduling units (bf16: CTA pairs, fp32: CTAs) that
// fit on the device at once.  Launchers take the number of units to run
// (each unit walks tiles unit, unit + units, ...; tile M blocks are
// GemmShape rows: 256 for bf16 pairs, 128 for fp32).
cudaError_t gemm_prepare_bf16(int sms, int* max_units);
cudaError_t gemm_prepare_fp32(int sms, int* max_units);

// Pass 1: A = X (K-major), B = W (K-major), epilogue = per-tile row statistics.
cudaError_t launch_logits_lse_bf16(const CUtensorMap& A, const CUtensorMap& B, const GemmGrid& g,
                                   const RowLseParams& p, int units, cudaStream_t s);
cudaError_t launch_logits_lse_fp32(const CUtensorMap& A, const CUtensorMap& B, const GemmGrid& g,
                                   const RowLseParams& p, int units, cudaStream_t s);
// Pass 2: A = X (K-major), B = W chunk (K-major), epilogue = G chunk store.
cudaError_t launch_logits_grad_bf16(const CUtensorMap& A, const CUtensorMap& B,
                                    const CUtensorMap& out, const GemmGrid& g,
                                    const GradLogitsParams& p, int units, cudaStream_t s);
cudaError_t launch_logits_grad_fp32(const CUtensorMap& A, const CUtensorMap& B,
                                    const CUtensorMap& out, const GemmGrid& g,
                                    const GradLogitsParams& p, int units, cudaStream_t s);
// dW chunk: A = G^T, B = X (bf16: both MN-major views of G and X; fp32:
// K-major transposed copies G^T [Vc, N] and X^T [H, N]), fp32 store.
cudaError_t launch_dw_bf16(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                           const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s);
cudaError_t launch_dw_fp32(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                           const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s);
// dX chunk: A = G (K-major), B = W chunk (bf16: MN-major view of W; fp32:
// K-major transposed copy W_c^T [H, Vc]), fp32 store or add.
cudaError_t launch_dx_bf16(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                           const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s);
cudaError_t launch_dx_fp32(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& out,
                           const GemmGrid& g, const StoreParams& p, int units, cudaStream_t s);

// Row combine: partial statistics -> lse2, row losses, mean loss, n_valid, scale.
struct CombineParams {
  const float* partial;   // [num_vblk][N]
  int32_t num_vblk;
  const float* st;        // [N]
  Targets target;         // [N]
  int64_t N;
  int64_t V;
  int64_t ignore_index;
  float* lse2;            // [N] (workspace)
  float* lse_out;         // optional [N]
  float* loss_rows_out;   // optional [N]
  double* blk_loss;       // [grid]
  int64_t* blk_cnt;       // [grid]
  Scalars* sc;
  float grad_scale;
  int64_t norm_count;
  float* loss_out;        // optional device
  int64_t* nvalid_out;    // optional device
};
constexpr int COMBINE_THREADS = 256;
int combine_grid(int64_t N);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);

// One block whose wait can never complete; it must expire after limit_ns.
cudaError_t launch_wait_expiry(Scalars* sc, uint64_t limit_ns, cudaStream_t s);

// Device status bits -> flce_status code in *out (one thread).
cudaError_t launch_status_code(const Scalars* sc, int32_t* out, cudaStream_t s);

// out[c * out_pitch + r] = in[r * in_pitch + c] for r < R, c < C, and 0 for
// R <= r < R_pad (fp32).
cudaError_t launch_transpose_f32(const float* in, int64_t R, int64_t C, int64_t in_pitch,
                                 float* out, int64_t out_pitch, int64_t R_pad, int sms,
                                 cudaStream_t s);

// Cross-entropy on materialised logits.
struct CeRowsParams {
  const void* logits;     // [N, V] bf16 or fp32
  void* dlogits;          // [N, V] same type, may equal logits; NULL = loss only
  Targets target;         // [N]
  int64_t N;
  int64_t V;
  int64_t ignore_index;
  const Scalars* sc;      // n_valid counted by launch_ce_count
  float grad_scale;
  int64_t norm_count;
  float* partial;         // [N] lse2 per row (the combine's single statistic)
  float* st;              // [N] target logit
  int32_t vectorized;     // rows start 16-byte aligned, V * elt % 16 == 0, < 2^30 vectors
};
cudaError_t launch_ce_count(Targets target, int64_t N, int64_t V, int64_t ignore_index,
                            Scalars* sc, int sms, cudaStream_t s);
cudaError_t launch_ce_rows(const CeRowsParams& p, int elt, int sms, cudaStream_t s);

// fp32 [n] -> bf16 [n] (round to nearest even).
cudaError_t launch_convert_bf16(const float* src, void* dst, int64_t n, int sms, cudaStream_t s);

// dst[i] = (dst type)(src[i] * *scale_dev) (scale 1 when scale_dev is NULL);
// element sizes 2 (bf16) or 4 (fp32).  In place when dst == src and the
// sizes are equal.
cudaError_t launch_scale_convert(const void* src, int src_elt, void* dst, int dst_elt, int64_t n,
                                 const float* scale_dev, int sms, cudaStream_t s);

}  // namespace flce
