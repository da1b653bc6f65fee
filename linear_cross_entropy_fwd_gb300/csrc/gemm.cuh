// gemm.cuh -- persistent, warp-specialised tcgen05 GEMM engine for sm_103a.
//
// D = A * B^T tile by tile, fp32 accumulation in TMEM, with a pluggable
// epilogue that reads the accumulator straight out of TMEM (so logits never
// travel to HBM).  Each scheduling unit (one CTA, or one CTA pair) walks the
// tile space tile = unit + i * units; the launch picks which tile index runs
// fastest (tile_coords) so the units that run together share tiles in L2.
//
// Launch overlap (programmatic dependent launch).  A launch's CTAs start as
// the previous launch's CTAs leave their SMs.  The producer and the MMA
// issuer start at once: they touch only operands written two or more
// launches back (or, with wait_operands set, the producer first waits for
// the previous launch).  The epilogue waits for the previous launch to
// complete before its first global access, then lets the next launch start.
// So when a launch starts, the one two before it has completed, and its
// early units run their first tiles' MMAs in the previous launch's tail.
// (Pass 2 follows the combine kernel, which lets it start at once: its
// operands are the inputs X and W, and its epilogue waits for the combine,
// which waits for pass 1.)
//
// Two shapes of the engine:
//   PAIR = false  one CTA per 128 x 256 tile (cta_group::1), 4-stage ring of
//                 48 KB stages (A 128 rows, B 256 rows, 128 bytes of K).
//   PAIR = true   a cluster of two CTAs per 256 x 256 tile (cta_group::2):
//                 each CTA stages its own 128 rows of A and half of B (128
//                 rows), the even CTA issues the MMAs for both, each CTA's
//                 TMEM holds its 128 accumulator rows.  6-stage ring of 32 KB
//                 stages; half the B traffic per SM of the single-CTA shape.
//
// Roles (192 threads per CTA):
//   warp 0      TMA producer
//   warp 1      TMEM allocator and MMA issuer (one thread of the even CTA),
//               two accumulators of BN fp32 columns so the epilogue of tile i
//               overlaps the MMAs of tile i+1
//   warps 2..5  epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, i.e. one
//               accumulator row per thread
//
// Operand layouts (both staged with the 128-byte swizzle that TMA writes):
//   K-major   rows of 128 bytes of K, 8-row groups 1024 bytes apart
//             (SBO = 1024); the k-th MMA of a stage starts 32*k bytes in.
//   MN-major  boxes of (128 bytes of MN) x (128/elt K rows), one box per
//             128 bytes of MN, boxes LBO = box bytes apart, 8 K rows 1024
//             bytes apart (SBO); the k-th MMA starts 32/elt*128*k bytes in.
#pragma once
#include "sm103.cuh"

namespace flce {

template <int ELT>
struct ElemTraits;
template <>
struct ElemTraits<2> {  // bf16 operands, kind::f16
  static constexpr uint32_t kFormat = 1;
  static constexpr int kStageK = 64;  // K elements per stage (128 bytes)
};
template <>
struct ElemTraits<4> {  // fp32 operands, kind::tf32
  static constexpr uint32_t kFormat = 2;
  static constexpr int kStageK = 32;
};

template <bool PAIR>
struct EngineShape {
  static constexpr int kCtas = PAIR ? 2 : 1;
  static constexpr int kBRows = BN / kCtas;  // rows of B staged per CTA
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr uint32_t kABytes = BM * 128;
  static constexpr uint32_t kBBytes = kBRows * 128;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static_assert(kStages * kStageBytes + STAGING_BYTES + SMEM_BARRIER_BYTES + 1024 <=
                    GEMM_SMEM_BYTES,
                "shared memory plan");
};

template <int ELT, bool A_MN, bool B_MN, bool PAIR, class Epi>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmOut, const GemmGrid g,
                const typename Epi::Params ep) {
  static_assert(!PAIR || ELT == 2, "CTA pairs are used for bf16 operands");
  using S = EngineShape<PAIR>;
  constexpr int STG = S::kStages;
  constexpr int KE = ElemTraits<ELT>::kStageK;
  constexpr uint32_t BOX_BYTES = 128u * KE;  // one MN-major box
  constexpr uint32_t IDESC =
      make_idesc(ElemTraits<ELT>::kFormat, A_MN, B_MN, BM * S::kCtas, BN);
  // start-address advance of the k-th MMA (K = 32 bytes) inside a stage
  constexpr uint32_t A_ADV = A_MN ? (32u / ELT) * 128u : 32u;
  constexpr uint32_t B_ADV = B_MN ? (32u / ELT) * 128u : 32u;
  constexpr uint32_t A_LBO = A_MN ? BOX_BYTES : 0u;
  constexpr uint32_t B_LBO = B_MN ? BOX_BYTES : 0u;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STG * S::kABytes;
  uint8_t* staging = smB + STG * S::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + STAGING_BYTES);
  uint64_t* full = bars;                // [STG]  (the even CTA's are the ones used)
  uint64_t* empty = bars + STG;         // [STG]
  uint64_t* acc_full = bars + 2 * STG;  // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]    (the even CTA's are the ones used)
  uint64_t* drain = acc_empty + 2;      // [1]
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int num_tiles = g.num_m_blk * g.num_n_blk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STG; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], EPI_WARPS * S::kCtas);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_base_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_base_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers exist before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_slot;
  // Everything above touched only this CTA's shared memory and TMEM, so it
  // overlaps the previous launch's tail.  From here each role waits for the
  // previous launch (griddepcontrol.wait) before it touches memory that
  // launch writes or reads.

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t gk = 0;
      bool ok = true;
      const uint64_t pol_a = l2_policy(g.a_l2);
      const uint64_t pol_b = l2_policy(g.b_l2);
      if (g.wait_operands) grid_dependency_wait();
      for (int tile = unit; ok && tile < num_tiles; tile += units) {
        int mu, n_blk;
        tile_coords(g, tile, mu, n_blk);
        const int m_blk = mu * S::kCtas + static_cast<int>(rank);
        const int a_mn = g.a_mn_off + m_blk * BM;
        const int b_mn = g.b_mn_off + n_blk * BN + static_cast<int>(rank) * S::kBRows;
        for (int kb = 0; kb < g.num_k_blk; ++kb, ++gk) {
          const uint32_t s = gk % STG;
          const uint32_t r = gk / STG;
          if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, g.status)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full[s], S::kCtas * S::kStageBytes);
          uint8_t* a_dst = smA + s * S::kABytes;
          uint8_t* b_dst = smB + s * S::kBBytes;
          const int ak = g.a_k_off + kb * KE;
          const int bk = g.b_k_off + kb * KE;
          if (PAIR) {
            const uint32_t fb = mapa_shared(smem_addr(&full[s]), 0);
            if (A_MN) {
#pragma unroll
              for (int j = 0; j < BM / KE; ++j)
                tma_load_2d_pair(&tmA, fb, a_dst + j * BOX_BYTES, a_mn + j * KE, ak);
            } else if (g.a_l2) {
              tma_load_2d_pair_hint(&tmA, fb, a_dst, ak, a_mn, pol_a);
            } else {
              tma_load_2d_pair(&tmA, fb, a_dst, ak, a_mn);
            }
            if (B_MN) {
#pragma unroll
              for (int j = 0; j < S::kBRows / KE; ++j)
                tma_load_2d_pair(&tmB, fb, b_dst + j * BOX_BYTES, b_mn + j * KE, bk);
            } else if (g.b_l2) {
              tma_load_2d_pair_hint(&tmB, fb, b_dst, bk, b_mn, pol_b);
            } else {
              tma_load_2d_pair(&tmB, fb, b_dst, bk, b_mn);
            }
          } else {
            if (A_MN) {
#pragma unroll
              for (int j = 0; j < BM / KE; ++j)
                tma_load_2d_hint(&tmA, &full[s], a_dst + j * BOX_BYTES, a_mn + j * KE, ak,
                                 pol_a);
            } else {
              tma_load_2d_hint(&tmA, &full[s], a_dst, ak, a_mn, pol_a);
            }
            if (B_MN) {
#pragma unroll
              for (int j = 0; j < S::kBRows / KE; ++j)
                tma_load_2d_hint(&tmB, &full[s], b_dst + j * BOX_BYTES, b_mn + j * KE, bk,
                                 pol_b);
            } else {
              tma_load_2d_hint(&tmB, &full[s], b_dst, bk, b_mn, pol_b);
            }
          }
        }
      }
      // Drain: every stage this thread loaded must have landed before exit.
      // The even CTA sees its loads land on `full`; the odd CTA's loads land
      // on the even CTA's barrier, so it waits until the MMAs released them.
      const uint32_t n_drain = gk < STG ? gk : STG;
      for (uint32_t i = 0; i < n_drain; ++i) {
        const uint32_t q = gk - 1 - i;
        if (rank == 0)
          mbar_wait_drain(&full[q % STG], (q / STG) & 1);
        else
          mbar_wait_drain(&empty[q % STG], (q / STG) & 1);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0 && rank == 0) {
      uint32_t gk = 0, it = 0;
      bool ok = true;
      const uint32_t a_base = smem_addr(smA);
      const uint32_t b_base = smem_addr(smB);
      for (int tile = unit; ok && tile < num_tiles; tile += units, ++it) {
        const uint32_t buf = it & 1;
        const uint32_t use = it >> 1;
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag, g.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < g.num_k_blk; ++kb, ++gk) {
          const uint32_t s = gk % STG;
          const uint32_t r = gk / STG;
          if (!mbar_wait(&full[s], r & 1, abort_flag, g.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = a_base + s * S::kABytes;
          const uint32_t b_addr = b_base + s * S::kBBytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t adesc = smem_desc_sw128(a_addr + k * A_ADV, A_LBO, 1024);
            const uint64_t bdesc = smem_desc_sw128(b_addr + k * B_ADV, B_LBO, 1024);
            const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
            if (PAIR)
              mma_f16_pair(d_tmem, adesc, bdesc, IDESC, acc);
            else if (ELT == 2)
              mma_f16(d_tmem, adesc, bdesc, IDESC, acc);
            else
              mma_tf32(d_tmem, adesc, bdesc, IDESC, acc);
          }
          // stage s is free (in both CTAs of a pair) once these MMAs read it
          if (PAIR)
            mma_commit_pair_mc(&empty[s], 0x3);
          else
            mma_commit(&empty[s]);
        }
        if (!ok) break;
        if (PAIR)
          mma_commit_pair_mc(&acc_full[buf], 0x3);  // accumulator buf complete
        else
          mma_commit(&acc_full[buf]);
      }
      // All MMAs issued by this thread have finished before TMEM is released.
      if (PAIR)
        mma_commit_pair(drain);
      else
        mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // The previous launch has completed before any epilogue reads or writes
    // global memory (and, through its own epilogue's wait, every launch
    // before it).  Then this CTA lets the next launch start: its CTAs take
    // SMs only as this launch's CTAs exit (the grid never has more units
    // than fit at once).
    grid_dependency_wait();
    if (warp == 2 && lane == 0) grid_launch_dependents();
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* stg = staging + (warp - 2) * 2 * STAGING_BUF_BYTES;
    uint32_t acc_empty_leader[2] = {0u, 0u};
    if (PAIR) {
      acc_empty_leader[0] = mapa_shared(smem_addr(&acc_empty[0]), 0);
      acc_empty_leader[1] = mapa_shared(smem_addr(&acc_empty[1]), 0);
    }
    typename Epi::State st;
    Epi::init(st);
    uint32_t it = 0;
    for (int tile = unit; tile < num_tiles; tile += units, ++it) {
      const uint32_t buf = it & 1;
      const uint32_t use = it >> 1;
      if (!mbar_wait(&acc_full[buf], use & 1, abort_flag, g.status)) break;
      tc_fence_after();
      int mu, n_blk;
      tile_coords(g, tile, mu, n_blk);
      const int m_blk = mu * S::kCtas + static_cast<int>(rank);
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + buf * BN;
      Epi::tile(ep, st, &tmOut, taddr, m_blk, n_blk, q, lane, stg);
      // every tcgen05.ld of this tile has completed (waited inside tile())
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(acc_empty_leader[buf]);
        else
          mbar_arrive(&acc_empty[buf]);
      }
    }
    if (lane == 0) bulk_wait<0>();  // TMA stores done before smem goes away
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // neither CTA leaves while the pair still uses it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace flce
