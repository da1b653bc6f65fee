// small_kernels.cu -- the bandwidth-bound steps of the path:
//   * row combine: per-tile row statistics -> lse, row loss, deterministic
//     mean loss, exact count of valid rows, gradient scale;
//   * fp32 -> bf16 conversion of the dX accumulator;
//   * fp32 transposes feeding the tf32 gradient GEMMs K-major operands.
#include <cuda_runtime.h>

#include "launch.h"
#include "sm103.cuh"

namespace flce {

constexpr float kLn2 = 0.69314718055994531f;

int combine_grid(int64_t N) {
  const int64_t b = (N + COMBINE_THREADS - 1) / COMBINE_THREADS;
  return b < 1 ? 1 : static_cast<int>(b);
}

// One thread per row.  lse2_i = M + log2(sum_b 2^(p_b - M)), M = max_b p_b,
// over the row's per-tile statistics p_b = m_b + log2(l_b) (pass 1).  The
// row loss is lse_i - S_{i,t_i} with lse_i = lse2_i ln 2.  Sums: per block a
// fixed shuffle tree in double, then the last block to finish adds the block
// sums in index order, so the result does not depend on scheduling.
__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const CombineParams p) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * COMBINE_THREADS + threadIdx.x;
  double row_loss = 0.0;
  int cnt = 0;
  if (i < p.N) {
    float m = -INFINITY, s = 0.f;
    const float* col = p.partial + i;
    int b = 0;
    for (; b + 4 <= p.num_vblk; b += 4) {
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = __ldg(col + static_cast<int64_t>(b + k) * p.N);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (v[k] > m) {
          s = s * fast_exp2(m - v[k]) + 1.f;
          m = v[k];
        } else {
          s += fast_exp2(v[k] - m);
        }
      }
    }
    for (; b < p.num_vblk; ++b) {
      const float v = __ldg(col + static_cast<int64_t>(b) * p.N);
      if (v > m) {
        s = s * fast_exp2(m - v) + 1.f;
        m = v;
      } else {
        s += fast_exp2(v - m);
      }
    }
    const float lse2 = m + fast_log2(s);
    p.lse2[i] = lse2;
    const float lse = lse2 * kLn2;
    if (p.lse_out) p.lse_out[i] = lse;
    const int64_t t = p.target[i];
    float lr = 0.f;
    if (t != p.ignore_index) {
      if (t < 0 || t >= p.V) {
        atomicOr(&p.sc->status, FLCE_DEV_TARGET);
      } else {
        lr = lse - p.st[i];
        cnt = 1;
      }
    }
    if (p.loss_rows_out) p.loss_rows_out[i] = lr;
    row_loss = lr;
  }
  // block reduction (fixed order)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    row_loss += __shfl_xor_sync(0xffffffffu, row_loss, off);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
  }
  __shared__ double s_loss[COMBINE_THREADS / 32];
  __shared__ int s_cnt[COMBINE_THREADS / 32];
  __shared__ bool s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_loss[warp] = row_loss;
    s_cnt[warp] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0;
    int64_t c = 0;
    for (int w = 0; w < COMBINE_THREADS / 32; ++w) {
      a += s_loss[w];
      c += s_cnt[w];
    }
    p.blk_loss[blockIdx.x] = a;
    p.blk_cnt[blockIdx.x] = c;
    __threadfence();
    const unsigned ticket = atomicAdd(&p.sc->ticket, 1u);
    s_last = (ticket == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  // last block: warp 0 adds the block sums in a fixed order
  __threadfence();
  double a = 0.0;
  int64_t c = 0;
  for (int b = lane; b < static_cast<int>(gridDim.x); b += 32) {
    a += __ldcg(p.blk_loss + b);
    c += __ldcg(reinterpret_cast<const long long*>(p.blk_cnt) + b);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    c += __shfl_xor_sync(0xffffffffu, c, off);
  }
  if (lane == 0) {
    const int64_t n = p.norm_count > 0 ? p.norm_count : c;
    const float loss = n > 0 ? static_cast<float>(a / static_cast<double>(n)) : 0.f;
    p.sc->loss_sum = a;
    p.sc->n_valid = c;
    p.sc->loss = loss;
    p.sc->scale = n > 0 ? static_cast<float>(static_cast<double>(p.grad_scale) /
                                             static_cast<double>(n))
                        : 0.f;
    p.sc->ticket = 0;
    if (p.loss_out) *p.loss_out = loss;
    if (p.nvalid_out) *p.nvalid_out = c;
  }
}

__global__ void status_code_kernel(const Scalars* sc, int32_t* out) {
  const int32_t bits = sc->status;
  // codes of the public flce_status enum: 7 = timeout, 4 = bad target
  *out = (bits & FLCE_DEV_TIMEOUT) ? 7 : ((bits & FLCE_DEV_TARGET) ? 4 : 0);
}

cudaError_t launch_status_code(const Scalars* sc, int32_t* out, cudaStream_t s) {
  status_code_kernel<<<1, 1, 0, s>>>(sc, out);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  combine_kernel<<<combine_grid(p.N), COMBINE_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

// 8 elements per thread and iteration (two 16-byte loads, one 16-byte store).
__global__ void convert_bf16_kernel(const float* __restrict__ src, uint4* __restrict__ dst,
                                    int64_t n8, const float* __restrict__ tail_src,
                                    uint16_t* __restrict__ tail_dst, int tail) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n8;
       k += stride) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(src) + 2 * k);
    const float4 b = __ldcs(reinterpret_cast<const float4*>(src) + 2 * k + 1);
    uint4 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    __stcs(dst + k, o);
  }
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail) {
    const uint32_t w = pack_bf16x2(tail_src[threadIdx.x], 0.f);
    tail_dst[threadIdx.x] = static_cast<uint16_t>(w & 0xFFFFu);
  }
}

cudaError_t launch_convert_bf16(const float* src, void* dst, int64_t n, int sms, cudaStream_t s) {
  const int64_t n8 = n / 8;
  const int tail = static_cast<int>(n - n8 * 8);
  int64_t blocks = (n8 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  convert_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      src, reinterpret_cast<uint4*>(dst), n8, src + n8 * 8,
      reinterpret_cast<uint16_t*>(dst) + n8 * 8, tail);
  return cudaGetLastError();
}

// 32 x 32 tiles through shared memory (one padding column: no bank conflicts).
__global__ void transpose_f32_kernel(const float* __restrict__ in, int64_t R, int64_t C,
                                     int64_t in_pitch, float* __restrict__ out,
                                     int64_t out_pitch, int64_t R_pad) {
  __shared__ float tile[32][33];
  const int64_t tiles_r = (R_pad + 31) / 32, tiles_c = (C + 31) / 32;
  for (int64_t t = blockIdx.x; t < tiles_r * tiles_c; t += gridDim.x) {
    const int64_t r0 = (t % tiles_r) * 32, c0 = (t / tiles_r) * 32;
    for (int k = threadIdx.y; k < 32; k += blockDim.y) {
      const int64_t r = r0 + k, c = c0 + threadIdx.x;
      tile[k][threadIdx.x] = (r < R && c < C) ? in[r * in_pitch + c] : 0.f;
    }
    __syncthreads();
    for (int k = threadIdx.y; k < 32; k += blockDim.y) {
      const int64_t c = c0 + k, r = r0 + threadIdx.x;
      if (c < C && r < R_pad) out[c * out_pitch + r] = tile[threadIdx.x][k];
    }
    __syncthreads();
  }
}

cudaError_t launch_transpose_f32(const float* in, int64_t R, int64_t C, int64_t in_pitch,
                                 float* out, int64_t out_pitch, int64_t R_pad, int sms,
                                 cudaStream_t s) {
  const int64_t tiles = ((R_pad + 31) / 32) * ((C + 31) / 32);
  int64_t blocks = tiles < static_cast<int64_t>(sms) * 16 ? tiles : static_cast<int64_t>(sms) * 16;
  if (blocks < 1) blocks = 1;
  transpose_f32_kernel<<<static_cast<unsigned>(blocks), dim3(32, 8), 0, s>>>(
      in, R, C, in_pitch, out, out_pitch, R_pad);
  return cudaGetLastError();
}

}  // namespace flce
