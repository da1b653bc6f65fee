// epilogues.cuh -- TMEM -> register epilogues of the fused linear
// cross-entropy GEMMs.  Each thread owns one accumulator row (one token row
// for the logit passes), so every row statistic is thread-local.
//
// Notation: S = X W^T (logits), lse2_i = log2 sum_j 2^(S_ij log2 e), so that
// lse_i = lse2_i ln 2 and softmax(S_i)_j = 2^(S_ij log2 e - lse2_i).
#pragma once
#include "gemm.cuh"

namespace flce {

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------------
// Pass 1 (logits -> per-tile row statistics).  For every row of the tile:
//   partial[n_blk][row] = m + log2(sum over the tile's columns of 2^(u - m)),
//   u = S * log2 e, m = max u  (columns >= V excluded),
// and, for the one tile that holds the row's target column, st[row] = S_{i,t_i}.
struct EpiRowLse {
  struct Params {
    Targets target;
    float* partial;   // [num_vocab_tiles][N]
    float* st;        // [N] target logit
    int64_t N;
    int64_t V;
    int32_t vtile_off;  // vocabulary tile of the launch's first tile column
  };
  struct State {};
  __device__ static void init(State&) {}

  __device__ static void tile(const Params& p, State&, const CUtensorMap*, uint32_t taddr,
                              int m_blk, int n_blk, int q, int lane, uint8_t*) {
    const int64_t row = static_cast<int64_t>(m_blk) * BM + 32 * q + lane;
    const int64_t vt = static_cast<int64_t>(n_blk) + p.vtile_off;  // global vocabulary tile
    const int64_t n0 = vt * BN;
    const int64_t rem = p.V - n0;
    const int valid_cols = rem < BN ? static_cast<int>(rem) : BN;
    const int64_t t = row < p.N ? p.target[row] : -1;
    const int64_t tl64 = t - n0;
    const int tcol = (tl64 >= 0 && tl64 < valid_cols) ? static_cast<int>(tl64) : -1;

    float m = -INFINITY, l = 0.f, st_val = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      if (32 * c >= valid_cols) break;  // warp-uniform
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + 32 * c, r);
      tmem_ld_wait();
      const int nv = valid_cols - 32 * c;  // >= 1
      float cmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nv) cmax = fmaxf(cmax, __uint_as_float(r[i]));
      const float mnew = fmaxf(m, cmax * kLog2e);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nv) acc += fast_exp2(fmaf(__uint_as_float(r[i]), kLog2e, -mnew));
      l = (m == -INFINITY ? 0.f : l * fast_exp2(m - mnew)) + acc;
      m = mnew;
      const int tl = tcol - 32 * c;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i == tl) st_val = __uint_as_float(r[i]);
    }
    if (row < p.N) {
      p.partial[vt * p.N + row] = m + fast_log2(l);
      if (tcol >= 0) p.st[row] = st_val;
    }
  }
};

// Staging helpers: a warp writes its 32 rows x 128 bytes into a 4 KB buffer
// in the 128-byte-swizzled layout TMA expects (16-byte chunk c of row r at
// chunk c ^ (r % 8)), then lane 0 hands it to the TMA unit.
struct Staging {
  uint32_t count;  // buffers handed out so far by this warp (alternates 0/1)
};

__device__ __forceinline__ uint8_t* staging_acquire(Staging& s, uint8_t* stg, int lane) {
  uint8_t* buf = stg + (s.count & 1) * STAGING_BUF_BYTES;
  ++s.count;
  if (lane == 0) bulk_wait_read<1>();  // the store that last read this buffer is done
  __syncwarp();
  return buf;
}

__device__ __forceinline__ void staging_put16(uint8_t* buf, int lane, int chunk, uint32_t a,
                                              uint32_t b, uint32_t c, uint32_t d) {
  const uint32_t addr = smem_addr(buf) + lane * 128 + ((chunk ^ (lane & 7)) << 4);
  st_shared_v4(addr, a, b, c, d);
}

template <bool REDUCE>
__device__ __forceinline__ void staging_release(const CUtensorMap* map, uint8_t* buf, int lane,
                                                int32_t x, int32_t y) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (REDUCE)
      tma_reduce_add_2d(map, buf, x, y);
    else
      tma_store_2d(map, buf, x, y);
    bulk_commit();
  }
}

// ------------------------------------------------------------------------
// Pass 2 (logits -> G chunk).  For the row's valid target t_i:
//   G_ij = (2^(S_ij log2 e - lse2_i) - [j == t_i]) * scale,  scale = grad_scale / n
// and 0 for ignored rows and for columns >= V.  Stored in the operand type
// (bf16 round-to-nearest-even, or fp32) to the chunk buffer [N, Vc].
template <int ELT>
struct EpiGradLogits {
  struct Params {
    Targets target;
    const float* lse2;          // [N]
    const Scalars* scalars;     // scale
    int64_t N;
    int64_t V;
    int64_t ignore_index;
    int64_t vocab_off;          // first vocabulary id of the chunk
  };
  using State = Staging;
  __device__ static void init(State& s) { s.count = 0; }

  __device__ static void tile(const Params& p, State& s, const CUtensorMap* out, uint32_t taddr,
                              int m_blk, int n_blk, int q, int lane, uint8_t* stg) {
    const int64_t row = static_cast<int64_t>(m_blk) * BM + 32 * q + lane;
    const int64_t col0 = p.vocab_off + static_cast<int64_t>(n_blk) * BN;  // vocab id
    bool valid = false;
    int64_t t = -1;
    float lse2 = 0.f;
    if (row < p.N) {
      t = p.target[row];
      valid = (t != p.ignore_index);
      lse2 = p.lse2[row];
    }
    const float scale = valid ? p.scalars->scale : 0.f;
    const int64_t tl64 = t - col0;
    const int tcol = (valid && tl64 >= 0 && tl64 < BN) ? static_cast<int>(tl64) : -1;
    const int64_t rem = p.V - col0;
    const int valid_cols = rem < BN ? static_cast<int>(rem) : BN;
    const int32_t y = m_blk * BM + 32 * q;
    constexpr int COLS = 128 / ELT;  // columns per 128-byte store box

#pragma unroll 1
    for (int u = 0; u < BN / COLS; ++u) {
      float v[COLS];
#pragma unroll
      for (int h = 0; h < COLS / 32; ++h) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + u * COLS + 32 * h, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * h + i] = __uint_as_float(r[i]);
      }
#pragma unroll
      for (int i = 0; i < COLS; ++i) {
        const int c = u * COLS + i;
        float gv = fast_exp2(fmaf(v[i], kLog2e, -lse2)) - (c == tcol ? 1.f : 0.f);
        gv = (c < valid_cols) ? gv * scale : 0.f;
        v[i] = gv;
      }
      uint8_t* buf = staging_acquire(s, stg, lane);
      if (ELT == 2) {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          staging_put16(buf, lane, ch, pack_bf16x2(v[8 * ch + 0], v[8 * ch + 1]),
                        pack_bf16x2(v[8 * ch + 2], v[8 * ch + 3]),
                        pack_bf16x2(v[8 * ch + 4], v[8 * ch + 5]),
                        pack_bf16x2(v[8 * ch + 6], v[8 * ch + 7]));
      } else {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          staging_put16(buf, lane, ch, __float_as_uint(v[4 * ch + 0]),
                        __float_as_uint(v[4 * ch + 1]), __float_as_uint(v[4 * ch + 2]),
                        __float_as_uint(v[4 * ch + 3]));
      }
      staging_release<false>(out, buf, lane, n_blk * BN + u * COLS, y);
    }
  }
};

// ------------------------------------------------------------------------
// Gradient GEMMs: the fp32 accumulator tile is stored (or added at L2 with
// a TMA reduction) to an fp32 [rows, H] output at (x_off + col, y_off + row).
struct EpiStoreF32 {
  struct Params {
    int32_t x_off;
    int32_t y_off;
    int32_t reduce;  // 0: overwrite, 1: out += tile
  };
  using State = Staging;
  __device__ static void init(State& s) { s.count = 0; }

  __device__ static void tile(const Params& p, State& s, const CUtensorMap* out, uint32_t taddr,
                              int m_blk, int n_blk, int q, int lane, uint8_t* stg) {
    const int32_t y = p.y_off + m_blk * BM + 32 * q;
#pragma unroll 1
    for (int u = 0; u < BN / 32; ++u) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + 32 * u, r);
      tmem_ld_wait();
      uint8_t* buf = staging_acquire(s, stg, lane);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        staging_put16(buf, lane, ch, r[4 * ch + 0], r[4 * ch + 1], r[4 * ch + 2], r[4 * ch + 3]);
      const int32_t x = p.x_off + n_blk * BN + 32 * u;
      if (p.reduce)
        staging_release<true>(out, buf, lane, x, y);
      else
        staging_release<false>(out, buf, lane, x, y);
    }
  }
};

}  // namespace flce
