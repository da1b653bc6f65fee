// flce_internal.h -- definitions shared by the host code and the kernels of
// libflce (not part of the public C ABI).
#pragma once
#include <cstddef>
#include <cstdint>

namespace flce {

// Bits of the per-call device status word.
enum : int32_t {
  FLCE_DEV_TARGET = 1,   // a target outside [0, V) that is not the ignore index
  FLCE_DEV_TIMEOUT = 2,  // a bounded wait inside a kernel expired
};

// GEMM tile: BM token/vocab rows x BN columns, K staged 128 bytes at a time.
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * 128;
constexpr int B_STAGE_BYTES = BN * 128;
constexpr int EPI_WARPS = 4;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int STAGING_BUF_BYTES = 4096;              // one 32-row x 128-byte TMA store box
constexpr int STAGING_BYTES = EPI_WARPS * 2 * STAGING_BUF_BYTES;
constexpr int TMEM_COLS = 2 * BN;                    // two fp32 accumulators of BN columns
constexpr int SMEM_BARRIER_BYTES = 256;
constexpr int GEMM_SMEM_BYTES =
    1024 + STAGES * (A_STAGE_BYTES + B_STAGE_BYTES) + STAGING_BYTES + SMEM_BARRIER_BYTES;

// Tile space and TMA coordinate offsets of one GEMM launch.
struct GemmGrid {
  int32_t num_m_blk;
  int32_t num_n_blk;
  int32_t num_k_blk;   // K blocks of 128 bytes
  int32_t a_mn_off;    // element offsets added to operand coordinates
  int32_t a_k_off;
  int32_t b_mn_off;
  int32_t b_k_off;
  int32_t raster_n;    // 0: M index fastest in the tile order, 1: N index fastest
  int32_t m_band;      // raster_n = 0 and 0 < m_band < num_m_blk: the tile order
                       // covers bands of m_band M blocks one after the other
  int32_t n_band;      // raster_n = 1 and 0 < n_band < num_n_blk: the same with
                       // bands of n_band N blocks (N fastest inside a band)
  int32_t a_l2;        // L2 policy of operand loads: 0 normal, 1 evict first,
  int32_t b_l2;        // 2 evict last
  int32_t wait_operands;  // 1: an operand is written by the launch just before
                          // this one, so the loads wait for it to complete
  int32_t* status;     // device status word (FLCE_DEV_* bits)
};

// Tile t of a launch -> (m block, n block).  The CTAs that run at the same
// time cover a band of consecutive tiles: the fastest index sweeps its whole
// operand, which should fit in L2 and stay resident, while the operand of
// the slow index streams through once.  With m_band, M runs fastest inside
// bands of m_band M blocks, and the bands follow one another: only one
// band's rows of the M operand need to stay in L2, and the N operand streams
// once per band.
__host__ __device__ inline void tile_coords(const GemmGrid& g, int tile, int& m_blk, int& n_blk) {
  if (g.raster_n && g.n_band > 0 && g.n_band < g.num_n_blk) {
    const int band_tiles = g.n_band * g.num_m_blk;
    const int band = tile / band_tiles;
    const int r = tile - band * band_tiles;
    const int n0 = band * g.n_band;
    const int cols = g.num_n_blk - n0 < g.n_band ? g.num_n_blk - n0 : g.n_band;
    n_blk = n0 + r % cols;
    m_blk = r / cols;
  } else if (g.raster_n) {
    n_blk = tile % g.num_n_blk;
    m_blk = tile / g.num_n_blk;
  } else if (g.m_band > 0 && g.m_band < g.num_m_blk) {
    const int band_tiles = g.m_band * g.num_n_blk;
    const int band = tile / band_tiles;
    const int r = tile - band * band_tiles;
    const int m0 = band * g.m_band;
    const int rows = g.num_m_blk - m0 < g.m_band ? g.num_m_blk - m0 : g.m_band;
    m_blk = m0 + r % rows;
    n_blk = r / rows;
  } else {
    m_blk = tile % g.num_m_blk;
    n_blk = tile / g.num_m_blk;
  }
}

// Target ids of a call: int64 (the default) or int32 [N], read as int64.
struct Targets {
  const void* p;
  int32_t is32;
  __host__ __device__ int64_t operator[](int64_t i) const {
    return is32 ? static_cast<int64_t>(static_cast<const int32_t*>(p)[i])
                : static_cast<const int64_t*>(p)[i];
  }
};

// Small device-side scalars of one call (cleared before its first kernel).
struct Scalars {
  int32_t status;
  uint32_t ticket;
  int64_t n_valid;
  float scale;        // grad_scale / normaliser (0 when nothing is valid)
  float loss;
  double loss_sum;
};

}  // namespace flce
