// gemm.cuh -- persistent, warp-specialised tcgen05 GEMM engine for sm_103a.
//
// D[BM x BN] = A[BM x K] * B[BN x K]^T per tile, fp32 accumulation in TMEM,
// with a pluggable epilogue that reads the accumulator straight out of TMEM
// (so logits never travel to HBM).  One CTA per SM walks the tile space
// tile = blockIdx.x + i * gridDim.x with the M index fastest, so the CTAs
// that run together share each B tile through L2.
//
// Roles (192 threads):
//   warp 0      TMA producer: STAGES-deep ring of A/B stages (128 bytes of K)
//   warp 1      TMEM allocator and MMA issuer (one thread), two accumulators
//               of BN fp32 columns so the epilogue of tile i overlaps the
//               MMAs of tile i+1
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

template <int ELT, bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmOut, const GemmGrid g,
                const typename Epi::Params ep) {
  constexpr int KE = ElemTraits<ELT>::kStageK;
  constexpr uint32_t BOX_BYTES = 128u * KE;  // one MN-major box
  constexpr uint32_t IDESC = make_idesc(ElemTraits<ELT>::kFormat, A_MN, B_MN, BM, BN);
  // start-address advance of the k-th MMA (K = 32 bytes) inside a stage
  constexpr uint32_t A_ADV = A_MN ? (32u / ELT) * 128u : 32u;
  constexpr uint32_t B_ADV = B_MN ? (32u / ELT) * 128u : 32u;
  constexpr uint32_t A_LBO = A_MN ? BOX_BYTES : 0u;
  constexpr uint32_t B_LBO = B_MN ? BOX_BYTES : 0u;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STAGES * A_STAGE_BYTES;
  uint8_t* staging = smB + STAGES * B_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + STAGING_BYTES);
  uint64_t* full = bars;                    // [STAGES]
  uint64_t* empty = bars + STAGES;          // [STAGES]
  uint64_t* acc_full = bars + 2 * STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint64_t* drain = acc_empty + 2;          // [1]
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = g.num_m_blk * g.num_n_blk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], EPI_WARPS);
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
    tmem_alloc(tmem_base_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t gk = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int m_blk = tile % g.num_m_blk;
        const int n_blk = tile / g.num_m_blk;
        const int a_mn = g.a_mn_off + m_blk * BM;
        const int b_mn = g.b_mn_off + n_blk * BN;
        for (int kb = 0; kb < g.num_k_blk; ++kb, ++gk) {
          const uint32_t s = gk % STAGES;
          const uint32_t r = gk / STAGES;
          if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, g.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], A_STAGE_BYTES + B_STAGE_BYTES);
          uint8_t* a_dst = smA + s * A_STAGE_BYTES;
          uint8_t* b_dst = smB + s * B_STAGE_BYTES;
          if (A_MN) {
#pragma unroll
            for (int j = 0; j < BM / KE; ++j)
              tma_load_2d(&tmA, &full[s], a_dst + j * BOX_BYTES, a_mn + j * KE,
                          g.a_k_off + kb * KE);
          } else {
            tma_load_2d(&tmA, &full[s], a_dst, g.a_k_off + kb * KE, a_mn);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < BN / KE; ++j)
              tma_load_2d(&tmB, &full[s], b_dst + j * BOX_BYTES, b_mn + j * KE,
                          g.b_k_off + kb * KE);
          } else {
            tma_load_2d(&tmB, &full[s], b_dst, g.b_k_off + kb * KE, b_mn);
          }
        }
      }
      // Drain: every stage this thread armed must have landed before exit.
      const uint32_t n_drain = gk < STAGES ? gk : STAGES;
      for (uint32_t i = 0; i < n_drain; ++i) {
        const uint32_t q = gk - 1 - i;
        mbar_wait_drain(&full[q % STAGES], (q / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      uint32_t gk = 0, it = 0;
      bool ok = true;
      const uint32_t a_base = smem_addr(smA);
      const uint32_t b_base = smem_addr(smB);
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++it) {
        const uint32_t buf = it & 1;
        const uint32_t use = it >> 1;
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag, g.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < g.num_k_blk; ++kb, ++gk) {
          const uint32_t s = gk % STAGES;
          const uint32_t r = gk / STAGES;
          if (!mbar_wait(&full[s], r & 1, abort_flag, g.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = a_base + s * A_STAGE_BYTES;
          const uint32_t b_addr = b_base + s * B_STAGE_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t adesc = smem_desc_sw128(a_addr + k * A_ADV, A_LBO, 1024);
            const uint64_t bdesc = smem_desc_sw128(b_addr + k * B_ADV, B_LBO, 1024);
            const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
            if (ELT == 2)
              mma_f16(d_tmem, adesc, bdesc, IDESC, acc);
            else
              mma_tf32(d_tmem, adesc, bdesc, IDESC, acc);
          }
          mma_commit(&empty[s]);  // stage s is free once these MMAs have read it
        }
        if (!ok) break;
        mma_commit(&acc_full[buf]);  // accumulator buf is complete
      }
      // All MMAs issued by this thread have finished before TMEM is released.
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* stg = staging + (warp - 2) * 2 * STAGING_BUF_BYTES;
    typename Epi::State st;
    Epi::init(st);
    uint32_t it = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
      const uint32_t buf = it & 1;
      const uint32_t use = it >> 1;
      if (!mbar_wait(&acc_full[buf], use & 1, abort_flag, g.status)) break;
      tc_fence_after();
      const int m_blk = tile % g.num_m_blk;
      const int n_blk = tile / g.num_m_blk;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + buf * BN;
      Epi::tile(ep, st, &tmOut, taddr, m_blk, n_blk, q, lane, stg);
      // every tcgen05.ld of this tile has completed (waited inside tile())
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    if (lane == 0) bulk_wait<0>();  // TMA stores done before smem goes away
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace flce
