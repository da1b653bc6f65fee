// small_kernels.cu -- the bandwidth-bound steps of the path:
//   * row combine: per-tile row statistics -> lse, row loss, deterministic
//     mean loss, exact count of valid rows, gradient scale;
//   * fp32 -> bf16 conversion of the dX accumulator;
//   * fp32 transposes feeding the tf32 gradient GEMMs K-major operands;
//   * cross-entropy on logits already materialised in memory: a count of
//     the valid rows, then one CTA per row computing the row statistics and
//     writing the gradient from a second read of the row (L2 eviction hints
//     keep the row resident between the two reads).
#include <cuda_runtime.h>

#include "launch.h"
#include "sm103.cuh"

namespace flce {

constexpr float kLn2 = 0.69314718055994531f;

// Online log2-domain sum: (m, l) holds max u and sum 2^(u - m).
__device__ __forceinline__ void online_add(float& m, float& l, float u) {
  // u in the log2 domain (logit * log2 e)
  if (u > m) {
    l = l * fast_exp2(m - u) + 1.f;
    m = u;
  } else if (u != -INFINITY) {  // a masked (-inf) logit adds nothing, even while m is -inf
    l += fast_exp2(u - m);
  }
}

__device__ __forceinline__ void online_merge(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  l = (m == -INFINITY ? 0.f : l * fast_exp2(m - M)) + (m2 == -INFINITY ? 0.f : l2 * fast_exp2(m2 - M));
  m = M;
}

// Rows per combine block: one per lane; the block's warps split the row's
// vocabulary tiles (warp w takes tiles w, w + COMBINE_SPLIT, ...), so every
// warp load reads 32 consecutive rows of one tile (128 contiguous bytes).
constexpr int COMBINE_ROWS = 32;
constexpr int COMBINE_SPLIT = COMBINE_THREADS / 32;

int combine_grid(int64_t N) {
  const int64_t b = (N + COMBINE_ROWS - 1) / COMBINE_ROWS;
  return b < 1 ? 1 : static_cast<int>(b);
}

// lse2_i = M + log2(sum_b 2^(p_b - M)), M = max_b p_b, over the row's per-tile
// statistics p_b = m_b + log2(l_b) (pass 1).  Each warp folds its share of
// the tiles with an online max/sum; the shares are merged in warp order.
// The row loss is lse_i - S_{i,t_i} with lse_i = lse2_i ln 2.  Sums: per
// block a fixed shuffle tree in double, then the last block to finish adds
// the block sums in index order, so the result does not depend on scheduling.
__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const CombineParams p) {
  // Launched to overlap the previous launch's tail; it reads that launch's
  // statistics only after its own wait.  The next launch may start at once.
  // In the bf16 fused path that is pass 2: before its own wait it reads only
  // X and W, which no kernel writes, and its first read of this kernel's
  // results comes after that wait (which ends once this kernel, and so pass
  // 1, has completed).  So pass 2's first tiles can run on the units pass
  // 1's last wave leaves idle.  Every other launch that follows this kernel
  // is a plain one, which starts only once this kernel has completed.
  grid_launch_dependents();
  grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * COMBINE_ROWS + lane;
  __shared__ float s_m[COMBINE_SPLIT][COMBINE_ROWS], s_l[COMBINE_SPLIT][COMBINE_ROWS];
  __shared__ bool s_last;
  {
    float m = -INFINITY, l = 0.f;
    if (i < p.N) {
      const float* col = p.partial + i;
      int b = warp;
      for (; b + 3 * COMBINE_SPLIT < p.num_vblk; b += 4 * COMBINE_SPLIT) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[k] = __ldg(col + static_cast<int64_t>(b + k * COMBINE_SPLIT) * p.N);
#pragma unroll
        for (int k = 0; k < 4; ++k) online_add(m, l, v[k]);
      }
      for (; b < p.num_vblk; b += COMBINE_SPLIT)
        online_add(m, l, __ldg(col + static_cast<int64_t>(b) * p.N));
    }
    s_m[warp][lane] = m;
    s_l[warp][lane] = l;
  }
  __syncthreads();
  double row_loss = 0.0;
  int cnt = 0;
  if (warp == 0 && i < p.N) {
    float m = s_m[0][lane], l = s_l[0][lane];
#pragma unroll
    for (int w = 1; w < COMBINE_SPLIT; ++w) online_merge(m, l, s_m[w][lane], s_l[w][lane]);
    const float lse2 = m + fast_log2(l);
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
  // block reduction (fixed order): warp 0 holds the block's rows
  if (warp == 0) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      row_loss += __shfl_xor_sync(0xffffffffu, row_loss, off);
      cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    }
    if (lane == 0) {
      p.blk_loss[blockIdx.x] = row_loss;
      p.blk_cnt[blockIdx.x] = cnt;
      __threadfence();
      const unsigned ticket = atomicAdd(&p.sc->ticket, 1u);
      s_last = (ticket == gridDim.x - 1);
    }
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

// Self-test of the bounded wait: one block waits on an mbarrier that nothing
// will ever arrive on; the wait must expire after limit_ns, record
// FLCE_DEV_TIMEOUT and let the kernel finish normally.
__global__ void wait_expiry_kernel(Scalars* sc, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, &abort_flag, &sc->status, limit_ns);
}

cudaError_t launch_wait_expiry(Scalars* sc, uint64_t limit_ns, cudaStream_t s) {
  wait_expiry_kernel<<<1, 32, 0, s>>>(sc, limit_ns);
  return cudaGetLastError();
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

// A launch that may begin while the previous one on the stream finishes
// (programmatic dependent launch); the kernel waits before it reads.
template <typename... Args>
cudaError_t launch_overlapped(void (*kernel)(Args...), unsigned blocks, unsigned threads,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  return launch_overlapped(combine_kernel, static_cast<unsigned>(combine_grid(p.N)),
                           COMBINE_THREADS, s, p);
}

// 8 elements per thread and iteration (two 16-byte loads, one 16-byte store).
__global__ void convert_bf16_kernel(const float* __restrict__ src, uint4* __restrict__ dst,
                                    int64_t n8, const float* __restrict__ tail_src,
                                    uint16_t* __restrict__ tail_dst, int tail) {
  grid_dependency_wait();  // the source is complete (overlapped launch)
  grid_launch_dependents();
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
  return launch_overlapped(convert_bf16_kernel, static_cast<unsigned>(blocks), 256u, s, src,
                           reinterpret_cast<uint4*>(dst), n8, src + n8 * 8,
                           reinterpret_cast<uint16_t*>(dst) + n8 * 8, tail);
}

// dst = (dst type)(src * scale), 8 elements per thread and iteration when both
// buffers are 16-byte aligned (the tail, or everything otherwise, one by one).
template <int SE, int DE>
__device__ __forceinline__ void load8(const void* src, int64_t k, float* f) {
  if (SE == 4) {
    const float4 a = __ldcs(static_cast<const float4*>(src) + 2 * k);
    const float4 b = __ldcs(static_cast<const float4*>(src) + 2 * k + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
    const uint4 u = __ldcs(static_cast<const uint4*>(src) + k);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __uint_as_float(w[e] << 16);
      f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
}

template <int SE, int DE>
__global__ void scale_convert_kernel(const void* __restrict__ src, void* __restrict__ dst,
                                     int64_t n, int vec, const float* __restrict__ scale_dev) {
  const float sc = scale_dev ? *scale_dev : 1.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n8 = vec ? n / 8 : 0;
  for (int64_t k = tid; k < n8; k += stride) {
    float f[8];
    load8<SE, DE>(src, k, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] *= sc;
    if (DE == 4) {
      __stcs(static_cast<float4*>(dst) + 2 * k, make_float4(f[0], f[1], f[2], f[3]));
      __stcs(static_cast<float4*>(dst) + 2 * k + 1, make_float4(f[4], f[5], f[6], f[7]));
    } else {
      __stcs(static_cast<uint4*>(dst) + k,
             make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                        pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7])));
    }
  }
  for (int64_t i = n8 * 8 + tid; i < n; i += stride) {
    const float x = (SE == 4 ? static_cast<const float*>(src)[i]
                             : __uint_as_float(static_cast<uint32_t>(
                                   static_cast<const uint16_t*>(src)[i]) << 16)) * sc;
    if (DE == 4)
      static_cast<float*>(dst)[i] = x;
    else
      static_cast<uint16_t*>(dst)[i] = static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xFFFFu);
  }
}

cudaError_t launch_scale_convert(const void* src, int src_elt, void* dst, int dst_elt, int64_t n,
                                 const float* scale_dev, int sms, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) ==
                  0;
  const int64_t work = vec ? (n + 7) / 8 : n;
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (src_elt == 4 && dst_elt == 4)
    scale_convert_kernel<4, 4><<<grid, 256, 0, s>>>(src, dst, n, vec, scale_dev);
  else if (src_elt == 4)
    scale_convert_kernel<4, 2><<<grid, 256, 0, s>>>(src, dst, n, vec, scale_dev);
  else if (dst_elt == 4)
    scale_convert_kernel<2, 4><<<grid, 256, 0, s>>>(src, dst, n, vec, scale_dev);
  else
    scale_convert_kernel<2, 2><<<grid, 256, 0, s>>>(src, dst, n, vec, scale_dev);
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

// ---------------------------------------------------------------------------
// Cross-entropy on materialised logits S [N, V] (bf16 or fp32).

// n_valid (atomic integer adds: exact) and the bad-target flag.
__global__ void ce_count_kernel(const Targets target, int64_t N, int64_t V,
                                int64_t ignore_index, Scalars* sc) {
  int cnt = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < N;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = target[i];
    if (t == ignore_index) continue;
    if (t < 0 || t >= V)
      atomicOr(&sc->status, FLCE_DEV_TARGET);
    else
      ++cnt;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
  if ((threadIdx.x & 31) == 0 && cnt)
    atomicAdd(reinterpret_cast<unsigned long long*>(&sc->n_valid),
              static_cast<unsigned long long>(cnt));
}

cudaError_t launch_ce_count(Targets target, int64_t N, int64_t V, int64_t ignore_index,
                            Scalars* sc, int sms, cudaStream_t s) {
  int64_t blocks = (N + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 4) blocks = static_cast<int64_t>(sms) * 4;
  if (blocks < 1) blocks = 1;
  ce_count_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(target, N, V, ignore_index, sc);
  return cudaGetLastError();
}

template <int ELT>
struct CeVec;
template <>
struct CeVec<2> {  // 8 bf16 per 16-byte access
  static constexpr int kPer = 8;
  static constexpr uint32_t kMaskedWord = 0xFF80FF80u;  // two bf16 -inf
  __device__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
  __device__ static float load1(const void* p, int64_t i) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16);
  }
  __device__ static void store1(void* p, int64_t i, float v) {
    static_cast<uint16_t*>(p)[i] = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
  }
};
template <>
struct CeVec<4> {  // 4 fp32 per 16-byte access
  static constexpr int kPer = 4;
  static constexpr uint32_t kMaskedWord = 0xFF800000u;  // fp32 -inf
  __device__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  __device__ static float load1(const void* p, int64_t i) {
    return static_cast<const float*>(p)[i];
  }
  __device__ static void store1(void* p, int64_t i, float v) { static_cast<float*>(p)[i] = v; }
};

// The row kernel keeps several rows in flight per SM (one per CTA) so that
// enough 16-byte loads are outstanding to run near the HBM copy rate.  Its
// second read of a row is an L2 hit only while the rows in flight fit in L2
// next to the gradient being written, so the first read marks its lines
// evict-last and the second read and the gradient stores evict-first.
// Without the hints the L2 hit rate of the second read was 6.9% (bf16
// 8192 x 128256): the kernel moved about 1.5x the algorithmic bytes.
//
// Threads per CTA, rows in flight (CTAs per SM) and 16-byte loads in flight
// per thread, by element size, measured on 8192 x 128256 logits (TB/s of
// algorithmic bytes):
//   bf16  512 x 2 x 5 4.89, 512 x 2 x 6 4.77-4.81, 512 x 2 x 4 4.77,
//         384 x 3 x 6 4.50, 512 x 3 x 4 4.50, 256 x 4 x 6 4.46,
//         768 x 2 x 4 4.30, 1024 x 1 x 4 4.03, 768 x 1 x 6 3.80;
//   fp32  1024 x 1 x 8 5.35, 1024 x 1 x 4 5.17, 512 x 1 x 8 4.89,
//         512 x 2 x 4 4.73, 256 x 2 x 8 4.61.
//
// kSplit CTAs (a cluster) share each row of 16-byte vectors.  Split rows are
// read from DRAM exactly once (8192 x 128256 bf16: 2.110 GB read for 2.10 GB
// of logits, against 2.50 GB with one CTA per row), but every row then waits
// on a cluster barrier.  Same-box sweep (TB/s of algorithmic bytes):
//   bf16  split 1: 512 x 2 x 5 5.01;  split 2: 512 x 2 x 5 4.57,
//         256 x 4 x 6 4.69, 256 x 4 x 8 4.13, 128 x 8 x 8 4.29;
//         split 4: 256 x 4 x 6 2.92, 128 x 8 x 6 3.48;
//   fp32  split 1: 1024 x 1 x 8 5.44;  split 2: 512 x 2 x 8 5.58,
//         512 x 2 x 5 4.66, 256 x 4 x 4 4.77, 128 x 8 x 4 4.55;
//         split 4: 256 x 4 x 6 4.14, 256 x 4 x 8 4.00.
// A 256 KB bf16 row is too short to pay for the barrier; a 512 KB fp32 row
// is not.
template <int ELT>
struct CeRowShape;
//
// kKeepBytes: the last bytes of a CTA's part of each row are also copied
// into shared memory during the first pass, and the gradient pass reads them
// from there: that part needs no second read from L2, and its first read is
// marked evict-first.  Same-box A/B (TB/s): bf16 keep 0 4.81, 64 KB 4.96,
// 96 KB 4.97; fp32 keep 0 5.35, 64 KB 5.31, 96 KB 5.48.  With 96 KB the bf16
// kernel reads 2.18 GB from DRAM for 2.10 GB of logits (2.50 GB without).
// 96 KB is also the most the two CTAs of an SM can hold without losing L1:
// at 2 x 96 KB the SM's shared memory fits a 196 KB carveout, above it the
// SM takes the largest one and L1 drops from about 60 to 28 KB, too little
// for the loads in flight.  Keeping 98.5 KB (an allocation of 98.5 or 106
// KB) cost 15%, and 104 or 110 KB with L1::no_allocate loads 11%.
// With the kept tail the loads in flight were swept again (same box, TB/s):
//   bf16  split 1, 512 x 2: depth 3 4.88, 4 5.00, 5 4.96, 6 4.89;
//         512 x 2 x 4 with 80 KB kept 4.97, 104 KB 4.68; 384 x 3 x 4 with
//         64 KB 4.85; 256 x 4 x 6 with 48 KB 4.02;
//   fp32  split 2, 512 x 2: depth 4 5.71, 5 5.97, 6 6.00, 7 5.91, 8 5.47,
//         10 5.69; 512 x 2 x 6 with 80 KB kept 5.95; 256 x 4 x 8 with
//         48 KB 4.05; split 1, 1024 x 1 x 8 with 192 KB 5.14.
// With the gradient pass cut to one comparison per vector for the target and
// the scale folded into the exponent (about half the instructions per
// logit), once more: bf16 512 x 2 depth 3 5.68, 4 5.87, 5 5.97, 6 5.55;
// fp32 split 2, 512 x 2 depth 4 5.90, 5 6.06, 6 6.02, 8 5.97.  More rows
// in flight with smaller kept tails, within the same carveout, lost again:
// bf16 256 x 4 x 5 with 48 KB 4.36, 384 x 3 x 4 with 64 KB 5.55 (6.03 for
// 512 x 2 x 5 on that box); fp32 4.14 and 5.48 (6.05).
#ifndef FLCE_CE_KEEP_BF16
#define FLCE_CE_KEEP_BF16 (96 * 1024)
#endif
#ifndef FLCE_CE_KEEP_FP32
#define FLCE_CE_KEEP_FP32 (96 * 1024)
#endif
template <>
struct CeRowShape<2> {
  static constexpr int kThreads = 512;
  static constexpr int kCtasPerSm = 2;
  static constexpr int kDepth = 5;
  static constexpr int kSplit = 1;
  static constexpr int kKeepBytes = FLCE_CE_KEEP_BF16;
};
template <>
struct CeRowShape<4> {
  static constexpr int kThreads = 512;
  static constexpr int kCtasPerSm = 2;
  static constexpr int kDepth = 5;
  static constexpr int kSplit = 2;
  static constexpr int kKeepBytes = FLCE_CE_KEEP_FP32;
};

// 16-byte global loads (read-only path, or coherent) with an L2 eviction
// policy that do not allocate the line in L1.
__device__ __forceinline__ uint4 ld_nc_na_hint(const uint4* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

__device__ __forceinline__ uint4 ld_na_hint(const uint4* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy)
               : "memory");
  return v;
}

// Row loads of the two passes: bf16 rows without allocating in L1 (same-box
// A/B +0.8 to +0.9% at 128256- and 152064-wide rows), fp32 rows as plain
// loads (the same setting cost them 0.6%).
template <int ELT>
__device__ __forceinline__ uint4 ce_ld_first(const uint4* p, uint64_t pol) {
  return ELT == 2 ? ld_nc_na_hint(p, pol) : ld_nc_hint(p, pol);
}
template <int ELT>
__device__ __forceinline__ uint4 ce_ld_second(const uint4* p, uint64_t pol) {
  return ELT == 2 ? ld_na_hint(p, pol) : ld_hint(p, pol);
}

// Folds NV 16-byte vectors into (m, l): the vectors' max first, so one
// rescale per call and then one exp2 and one add per element.
template <int ELT, int NV>
__device__ __forceinline__ void ce_stats_add(const uint4 (&u)[NV], float& m, float& l) {
  using Vec = CeVec<ELT>;
  constexpr float kLog2e = 1.4426950408889634f;
  float f[NV][Vec::kPer];
  float bmax = -INFINITY;
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    Vec::unpack(u[q], f[q]);
#pragma unroll
    for (int e = 0; e < Vec::kPer; ++e) bmax = fmaxf(bmax, f[q][e]);
  }
  const float um = bmax * kLog2e;
  if (um > m) {
    l *= fast_exp2(m - um);  // m = -inf: l is 0 and stays 0
    m = um;
  }
  // while every logit so far is -inf (masked), m is -inf and each term is 0
  const float sub = m == -INFINITY ? 0.f : m;
#pragma unroll
  for (int q = 0; q < NV; ++q)
#pragma unroll
    for (int e = 0; e < Vec::kPer; ++e) l += fast_exp2(fmaf(f[q][e], kLog2e, -sub));
}

// Pass A over one CTA's vectors k, k + T, ... below hi of a row: (m, l) in the
// log2 domain, kDepth 16-byte loads in flight per thread (also in the last,
// partial batch).  With KEEP each vector read is also copied to
// keep[kk - keep_off].
template <int ELT, bool KEEP>
__device__ __forceinline__ void ce_stats_vectors(const uint4* rv, int k, int hi, uint64_t pol,
                                                 uint4* keep, int keep_off, float& m, float& l) {
  constexpr int D = CeRowShape<ELT>::kDepth, T = CeRowShape<ELT>::kThreads;
  for (; k + (D - 1) * T < hi; k += D * T) {
    uint4 u[D];
#pragma unroll
    for (int q = 0; q < D; ++q) u[q] = ce_ld_first<ELT>(rv + k + q * T, pol);
    if (KEEP) {
#pragma unroll
      for (int q = 0; q < D; ++q) keep[k + q * T - keep_off] = u[q];
    }
    ce_stats_add<ELT, D>(u, m, l);
  }
  if (k < hi) {
    // the passes that remain (fewer than kDepth): their loads in flight
    // together; a vector past the end reads as -inf and adds nothing
    constexpr uint32_t kM = CeVec<ELT>::kMaskedWord;
    uint4 u[D];
#pragma unroll
    for (int q = 0; q < D; ++q)
      u[q] = k + q * T < hi ? ce_ld_first<ELT>(rv + k + q * T, pol) : make_uint4(kM, kM, kM, kM);
    if (KEEP) {
#pragma unroll
      for (int q = 0; q < D; ++q)
        if (k + q * T < hi) keep[k + q * T - keep_off] = u[q];
    }
    ce_stats_add<ELT, D>(u, m, l);
  }
}

// dS of one 16-byte vector: 2^(S log2 e - c) for every element, the target's
// element (te of vector tv) less `one`, then (unless FOLD) times sc.  With
// FOLD, c already holds lse2 - log2 sc and `one` is sc.
template <int ELT, bool FOLD>
__device__ __forceinline__ uint4 ce_grad_vector(const uint4& u, int kk, float c, float sc,
                                                float one, int tv, int te) {
  using Vec = CeVec<ELT>;
  constexpr float kLog2e = 1.4426950408889634f;
  float f[Vec::kPer];
  Vec::unpack(u, f);
#pragma unroll
  for (int e = 0; e < Vec::kPer; ++e) f[e] = fast_exp2(fmaf(f[e], kLog2e, -c));
  if (kk == tv) {  // one vector per row
#pragma unroll
    for (int e = 0; e < Vec::kPer; ++e)
      if (e == te) f[e] -= one;
  }
  if (!FOLD) {
#pragma unroll
    for (int e = 0; e < Vec::kPer; ++e) f[e] *= sc;
  }
  return Vec::pack(f);
}

// Pass B over one CTA's vectors k, k + T, ... below hi of a row: read from
// global memory (an L2 hit: the row was just read), or from keep[kk -
// keep_off] where pass A copied them; dS written to ov.  rv and ov may be the
// same row (in place): each thread reads a vector before it writes it.
template <int ELT, bool FROM_KEEP, bool FOLD>
__device__ __forceinline__ void ce_grad_vectors(const uint4* rv, uint4* ov, int k, int hi,
                                                const uint4* keep, int keep_off, uint64_t pol,
                                                float c, float sc, float one, int tv, int te) {
  constexpr int D = CeRowShape<ELT>::kDepth, T = CeRowShape<ELT>::kThreads;
  for (; k + (D - 1) * T < hi; k += D * T) {
    uint4 u[D];
#pragma unroll
    for (int q = 0; q < D; ++q)
      u[q] = FROM_KEEP ? keep[k + q * T - keep_off] : ce_ld_second<ELT>(rv + k + q * T, pol);
#pragma unroll
    for (int q = 0; q < D; ++q)
      st_hint(ov + k + q * T, ce_grad_vector<ELT, FOLD>(u[q], k + q * T, c, sc, one, tv, te),
              pol);
  }
  if (k < hi) {  // the passes that remain (fewer than kDepth), loads in flight together
    uint4 u[D];
#pragma unroll
    for (int q = 0; q < D; ++q) {
      u[q] = make_uint4(0u, 0u, 0u, 0u);
      if (k + q * T < hi)
        u[q] = FROM_KEEP ? keep[k + q * T - keep_off] : ce_ld_second<ELT>(rv + k + q * T, pol);
    }
#pragma unroll
    for (int q = 0; q < D; ++q)
      if (k + q * T < hi)
        st_hint(ov + k + q * T, ce_grad_vector<ELT, FOLD>(u[q], k + q * T, c, sc, one, tv, te),
                pol);
  }
}

template <int ELT, bool FOLD>
__device__ __forceinline__ void ce_grad_row(const uint4* rv, uint4* ov, int v_lo, int v_keep,
                                            int v_hi, const uint4* keep, uint64_t pol, float c,
                                            float sc, float one, int tv, int te) {
  ce_grad_vectors<ELT, false, FOLD>(rv, ov, v_lo + static_cast<int>(threadIdx.x), v_keep, keep,
                                    0, pol, c, sc, one, tv, te);
  ce_grad_vectors<ELT, true, FOLD>(rv, ov, v_keep + static_cast<int>(threadIdx.x), v_hi, keep,
                                   v_keep, pol, c, sc, one, tv, te);
}

// SPLIT CTAs per row (grid-stride over rows; SPLIT = 2 is a cluster of two
// CTAs, each taking one half of every row's 16-byte vectors).  Pass A: max
// and sum of 2^(S log2 e) per thread, merged across the CTA and, with SPLIT
// = 2, with the peer CTA's half through distributed shared memory (merged in
// rank order, so both CTAs hold the same lse); lse2 and the target logit go
// to the row-statistics buffers the combine kernel reads.  Pass B (when dS is
// wanted): the CTA's part of the row again, and dS = (2^(S log2 e - lse2) -
// [j = t]) * grad_scale / n, zero on a row whose target is ignored.
// Splitting a row halves the bytes each SM keeps pending in L2 between a
// row's two reads.
//
// On the vector path each row's part is two ranges: [v_lo, v_keep), read
// from global memory in both passes, and [v_keep, v_hi), at most kKeepBytes,
// which pass A also copies to shared memory and pass B reads from there.
// Each range is walked from its own start (thread t takes its vectors t, t +
// kThreads, ...), so neither tests a vector's position against v_keep, and
// each thread reads back from shared memory exactly the vectors it put
// there.  With a positive
// scale sc, pass B computes 2^(S log2 e - (lse2 - log2 sc)) instead of
// multiplying by sc, and corrects the target's element by -sc: the one
// vector of the row that holds it is found by one comparison per vector.
template <int ELT, int SPLIT>
__global__ void __launch_bounds__(CeRowShape<ELT>::kThreads, CeRowShape<ELT>::kCtasPerSm)
    ce_rows_kernel(const CeRowsParams p) {
  constexpr int kThreads = CeRowShape<ELT>::kThreads;
  using Vec = CeVec<ELT>;
  constexpr float kLog2e = 1.4426950408889634f;
  __shared__ float s_m[kThreads / 32], s_l[kThreads / 32];
  __shared__ float s_lse2;
  __shared__ float2 s_half[2];  // this CTA's (max, sum) of its part of the row, by row parity
  extern __shared__ uint4 s_keep[];  // the kept tail of this CTA's part of the row
  constexpr int kKeepVecs = CeRowShape<ELT>::kKeepBytes / 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = static_cast<int>(threadIdx.x);
  const bool vec = SPLIT > 1 || p.vectorized;  // split rows are always vectorised
  // vector indices within a row fit in an int: the host vectorises only rows
  // of fewer than 2^30 vectors
  const int nvec = vec ? static_cast<int>(p.V / Vec::kPer) : 0;
  const int rank = SPLIT > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int per_cta = (nvec + SPLIT - 1) / SPLIT;
  const int v_lo = rank * per_cta < nvec ? rank * per_cta : nvec;  // this CTA's vectors
  const int v_hi = v_lo + per_cta < nvec ? v_lo + per_cta : nvec;
  // vectors [v_keep, v_hi) stay in shared memory between the two passes
  // (only when there is a gradient pass and the rows are vectorised)
  int v_keep = v_hi;
  if (vec && p.dlogits) v_keep = v_hi - kKeepVecs > v_lo ? v_hi - kKeepVecs : v_lo;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) / SPLIT;
  const int64_t row_step = static_cast<int64_t>(gridDim.x) / SPLIT;
  const int64_t n = p.norm_count > 0 ? p.norm_count : p.sc->n_valid;
  const float scale = n > 0 ? static_cast<float>(static_cast<double>(p.grad_scale) /
                                                 static_cast<double>(n))
                            : 0.f;
  const bool fold = scale > 0.f;
  const float log2_scale = fold ? log2f(scale) : 0.f;
  const uint64_t pol_keep = l2_policy(p.dlogits ? 2 : 1), pol_stream = l2_policy(1);
  int parity = 0;
  for (int64_t r = row0; r < p.N; r += row_step, parity ^= 1) {
    const uint8_t* row = static_cast<const uint8_t*>(p.logits) + r * p.V * ELT;
    float m = -INFINITY, l = 0.f;
    if (vec) {
      const uint4* rv = reinterpret_cast<const uint4*>(row);
      ce_stats_vectors<ELT, false>(rv, v_lo + tid, v_keep, pol_keep, s_keep, 0, m, l);
      ce_stats_vectors<ELT, true>(rv, v_keep + tid, v_hi, pol_stream, s_keep, v_keep, m, l);
    } else {
      for (int64_t j = threadIdx.x; j < p.V; j += kThreads)
        online_add(m, l, Vec::load1(row, j) * kLog2e);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
      online_merge(m, l, m2, l2);
    }
    if (lane == 0) {
      s_m[warp] = m;
      s_l[warp] = l;
    }
    __syncthreads();
    float M = 0.f, L = 0.f;
    if (threadIdx.x == 0) {
      M = s_m[0];
      L = s_l[0];
      for (int w = 1; w < kThreads / 32; ++w) online_merge(M, L, s_m[w], s_l[w]);
    }
    if (SPLIT > 1) {
      // swap the halves' statistics with the peer CTA; the slot alternates
      // with the row, so the peer's read of this row's slot is ordered
      // before this CTA rewrites it (two rows later) by the next row's
      // cluster barrier
      if (threadIdx.x == 0) s_half[parity] = make_float2(M, L);
      cluster_sync();
      if (threadIdx.x == 0) {
        const uint32_t slot = smem_addr(&s_half[parity]);
        const float2 h0 = ld_shared_cluster_f2(mapa_shared(slot, 0));
        M = h0.x;
        L = h0.y;
#pragma unroll
        for (int k = 1; k < SPLIT; ++k) {
          const float2 hk = ld_shared_cluster_f2(mapa_shared(slot, static_cast<uint32_t>(k)));
          online_merge(M, L, hk.x, hk.y);
        }
      }
    }
    if (threadIdx.x == 0) {
      const float lse2 = M + fast_log2(L);
      s_lse2 = lse2;
      if (rank == 0) p.partial[r] = lse2;
      // the target logit, written by the CTA whose part holds it (rank 0
      // writes 0 for an ignored or out-of-range target)
      const int64_t t = p.target[r];
      const bool in_row = (t >= 0 && t < p.V);
      const int owner = (SPLIT > 1 && in_row) ? static_cast<int>(t / Vec::kPer / per_cta) : 0;
      if (rank == owner) p.st[r] = in_row ? Vec::load1(row, t) : 0.f;
    }
    __syncthreads();
    if (p.dlogits) {
      const float lse2 = s_lse2;
      const int64_t t = p.target[r];
      const bool valid = (t != p.ignore_index) && t >= 0 && t < p.V;
      uint8_t* out = static_cast<uint8_t*>(p.dlogits) + r * p.V * ELT;
      if (vec) {
        const uint4* rv = reinterpret_cast<const uint4*>(row);
        uint4* ov = reinterpret_cast<uint4*>(out);
        if (!valid) {
          for (int k = v_lo + tid; k < v_hi; k += kThreads)
            st_hint(ov + k, make_uint4(0u, 0u, 0u, 0u), pol_stream);
        } else {
          const int tv = static_cast<int>(t / Vec::kPer);
          const int te = static_cast<int>(t - static_cast<int64_t>(tv) * Vec::kPer);
          if (fold)
            ce_grad_row<ELT, true>(rv, ov, v_lo, v_keep, v_hi, s_keep, pol_stream,
                                   lse2 - log2_scale, scale, scale, tv, te);
          else
            ce_grad_row<ELT, false>(rv, ov, v_lo, v_keep, v_hi, s_keep, pol_stream, lse2, scale,
                                    1.f, tv, te);
        }
      } else {
        const float sc = valid ? scale : 0.f;
        for (int64_t j = threadIdx.x; j < p.V; j += kThreads) {
          const float x = Vec::load1(row, j);
          const float g =
              valid ? (fast_exp2(fmaf(x, kLog2e, -lse2)) - (j == t ? 1.f : 0.f)) * sc : 0.f;
          Vec::store1(out, j, g);
        }
      }
    }
    __syncthreads();  // s_m / s_l / s_lse2 / s_keep are reused by the next row
  }
}

template <int ELT, int SPLIT>
cudaError_t launch_ce_rows_t(const CeRowsParams& p, int sms, cudaStream_t s) {
  using Shape = CeRowShape<ELT>;
  const int64_t cap = static_cast<int64_t>(sms) * Shape::kCtasPerSm / SPLIT;  // rows in flight
  const int64_t rows = p.N < cap ? p.N : cap;
  const int keep = (p.vectorized && p.dlogits) ? Shape::kKeepBytes : 0;
  if (keep > 0) {
    const cudaError_t e = cudaFuncSetAttribute(
        ce_rows_kernel<ELT, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, keep);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(rows * SPLIT));
  cfg.blockDim = dim3(Shape::kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(keep);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = SPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ce_rows_kernel<ELT, SPLIT>, p);
}

cudaError_t launch_ce_rows(const CeRowsParams& p, int elt, int sms, cudaStream_t s) {
  if (p.N < 1) return cudaSuccess;
  // rows of whole 16-byte vectors may be split across a cluster
  if (p.vectorized)
    return elt == 2 ? launch_ce_rows_t<2, CeRowShape<2>::kSplit>(p, sms, s)
                    : launch_ce_rows_t<4, CeRowShape<4>::kSplit>(p, sms, s);
  return elt == 2 ? launch_ce_rows_t<2, 1>(p, sms, s) : launch_ce_rows_t<4, 1>(p, sms, s);
}

}  // namespace flce
