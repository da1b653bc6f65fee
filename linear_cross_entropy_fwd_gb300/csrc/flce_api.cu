// flce_api.cu -- host side of libflce: argument checks, the workspace plan,
// TMA descriptors, the launch sequence and the extern "C" entry points.
//
// Launch sequence of one call (all on the caller's stream, no host sync
// unless the call is synchronous):
//   1  logits_lse   pass 1: S tiles = X W^T in TMEM; per-tile row max/sum-exp
//   2  combine      lse_i, row loss, mean loss, n_valid, gradient scale
//   for each vocabulary chunk c = [c0, c0 + vc):
//   3  logits_grad  pass 2: recompute S[:, c] in TMEM, G_c = (softmax - onehot) * scale
//   4  dw           dW[c] = G_c^T X            (fp32, written once)
//   5  dx           dX_acc (+)= G_c W[c]       (fp32, TMA add at L2 after chunk 0)
//   6  convert      dX_acc -> dX (bf16 inputs only; fp32 inputs accumulate in dX)
// fp32 inputs (tf32 products) feed steps 4 and 5 K-major transposed copies
// X^T, G_c^T and W[c]^T made by a transpose kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/flce.h"
#include "launch.h"

namespace flce {
namespace {

thread_local char g_last_error[512] = {0};

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
}

int cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
  return FLCE_ERR_CUDA;
}

#define FLCE_CUDA(call)                                 \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ----------------------------------------------------------- device cache
struct DeviceInfo {
  int sms = 0;
  bool ok_arch = false;
  int units_bf16 = 0;  // resident CTA pairs of the bf16 GEMM kernels (0 = not prepared)
  int units_fp32 = 0;  // resident CTAs of the fp32 GEMM kernels (0 = not prepared)
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

int device_info(int dtype, DeviceInfo* out) {
  int dev = 0;
  FLCE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal %d out of range", dev);
    return FLCE_ERR_ARG;
  }
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (d.sms == 0) {
    int major = 0, minor = 0, sms = 0;
    FLCE_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    FLCE_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    FLCE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    d.ok_arch = (major == 10 && minor == 3);
    d.sms = sms;
    if (!d.ok_arch) {
      set_error("device %d has compute capability %d.%d; libflce is built for 10.3 (sm_103a)",
                dev, major, minor);
    }
  }
  if (!d.ok_arch) return FLCE_ERR_ARCH;
  if (dtype == FLCE_BF16 && d.units_bf16 == 0) FLCE_CUDA(gemm_prepare_bf16(d.sms, &d.units_bf16));
  if (dtype == FLCE_FP32 && d.units_fp32 == 0) FLCE_CUDA(gemm_prepare_fp32(d.sms, &d.units_fp32));
  *out = d;
  return FLCE_OK;
}

// ------------------------------------------------------- library memory pool
// Scratch the library allocates itself comes from one stream-ordered pool per
// device that keeps freed memory mapped (release threshold: unlimited), so a
// synchronous call does not re-map its scratch every time.  The pool holds at
// most the largest scratch of the calls made so far, until the process exits.
cudaMemPool_t g_pool[kMaxDevices] = {};
std::mutex g_pool_mutex;

int pool_alloc(void** p, size_t bytes, cudaStream_t s) {
  int dev = 0;
  FLCE_CUDA(cudaGetDevice(&dev));
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    if (!g_pool[dev]) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t np;
      FLCE_CUDA(cudaMemPoolCreate(&np, &props));
      uint64_t keep = UINT64_MAX;
      FLCE_CUDA(cudaMemPoolSetAttribute(np, cudaMemPoolAttrReleaseThreshold, &keep));
      g_pool[dev] = np;
    }
    pool = g_pool[dev];
  }
  FLCE_CUDA(cudaMallocFromPoolAsync(p, bytes, pool, s));
  return FLCE_OK;
}

// ------------------------------------------------------------ TMA encode
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2D map over a row-major [rows, cols] matrix: dim0 = cols (contiguous).
int make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elt, uint64_t cols,
             uint64_t rows, uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows,
             const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return FLCE_ERR_CUDA;
  }
  if (box_cols * static_cast<uint32_t>(elt) != 128u || box_rows == 0 || box_rows > 256) {
    set_error("internal: bad TMA box for %s", what);
    return FLCE_ERR_ARG;
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled(%s) failed with CUresult %d (cols=%llu rows=%llu pitch=%llu)",
              what, static_cast<int>(r), static_cast<unsigned long long>(cols),
              static_cast<unsigned long long>(rows), static_cast<unsigned long long>(pitch_bytes));
    return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

// ------------------------------------------------------------------ plan
struct Plan {
  int64_t N = 0, H = 0, V = 0;
  int dtype = FLCE_BF16;
  int elt = 2;
  bool grads = false;
  int64_t num_vblk = 0;   // vocabulary tiles of BN columns
  int64_t Vc = 0;         // chunk width (multiple of BN)
  int64_t num_chunks = 0;
  int cgrid = 1;          // combine blocks
  int64_t Np = 0;         // N rounded up to 4 (row pitch of the fp32 transposes)
  size_t off_sc = 0, off_blk_loss = 0, off_blk_cnt = 0, off_lse2 = 0, off_st = 0,
         off_partial = 0, off_dxacc = 0, off_xt = 0, off_G = 0, off_gt = 0, off_wt = 0,
         total = 0;
};

size_t fixed_bytes(Plan& p) {
  size_t o = 0;
  p.off_sc = o;
  o += align_up(sizeof(Scalars), 256);
  p.off_blk_loss = o;
  o += align_up(static_cast<size_t>(p.cgrid) * sizeof(double), 256);
  p.off_blk_cnt = o;
  o += align_up(static_cast<size_t>(p.cgrid) * sizeof(int64_t), 256);
  p.off_lse2 = o;
  o += align_up(static_cast<size_t>(p.N) * 4, 256);
  p.off_st = o;
  o += align_up(static_cast<size_t>(p.N) * 4, 256);
  p.off_partial = o;
  o += align_up(static_cast<size_t>(p.num_vblk) * static_cast<size_t>(p.N) * 4, 256);
  p.off_dxacc = o;
  if (p.grads && p.dtype == FLCE_BF16)
    o += align_up(static_cast<size_t>(p.N) * static_cast<size_t>(p.H) * 4, 256);
  p.off_xt = o;
  if (p.grads && p.dtype == FLCE_FP32)
    o += align_up(static_cast<size_t>(p.H) * static_cast<size_t>(p.Np) * 4, 256);
  p.off_G = o;
  return o;
}

constexpr int64_t kMinChunk = 2048;
// The default budget never goes below this: where one sixteenth of the
// logits is smaller, the fixed part alone (the fp32 dX accumulator) can
// exceed it and the chunk loop would be all launch overhead.
constexpr size_t kBudgetFloor = size_t{96} << 20;
// Scheduling units the planner assumes (GB300: 152 SMs = 76 CTA pairs), so
// that a plan, and flce_workspace_bytes(), do not depend on which device
// (if any) is current when it is made.
constexpr int64_t kPlanUnitsPair = 76, kPlanUnitsSingle = 152;
// Per-launch cost the planner charges (ramp-up, last epilogue, launch gap),
// in 128-byte K blocks of one tile (one K block of a pair tile is ~0.27 us):
// about 7 us, as measured between chunk widths 4864 and 6656.
constexpr int64_t kPlanLaunchCost = 26;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Estimated time of the chunk loop for chunk width Vc, in K blocks of one
// unit: each GEMM launch costs (waves of tiles) x (K blocks per tile) plus a
// fixed launch cost.  Captures wave quantisation: a chunk whose dW tiles fill
// 5.5 waves costs as much as 6.
int64_t chunk_loop_cost(int64_t N, int64_t H, int64_t V, int64_t Vc, int elt, bool pair) {
  const int64_t U = pair ? kPlanUnitsPair : kPlanUnitsSingle;
  const int64_t mb = pair ? 2 * BM : BM, ke = 128 / elt;
  const int64_t mp = ceil_div(N, mb), nh = ceil_div(H, BN);
  const int64_t kH = ceil_div(H, ke), kN = ceil_div(N, ke);
  int64_t cost = 0;
  for (int64_t c0 = 0; c0 < V; c0 += Vc) {
    const int64_t vc = (V - c0) < Vc ? (V - c0) : Vc;
    const int64_t nb = ceil_div(vc, BN);
    cost += ceil_div(mp * nb, U) * kH;                    // pass 2 (G chunk)
    cost += ceil_div(ceil_div(vc, mb) * nh, U) * kN;      // dW chunk
    cost += ceil_div(mp * nh, U) * ceil_div(vc, ke);      // dX chunk
    cost += 3 * kPlanLaunchCost;
    // chunks after the first add into the fp32 dX accumulator: 8 bytes of
    // traffic per element, partly hidden under the MMAs (about 70 K blocks
    // at N x H = 8192 x 4096, in proportion elsewhere)
    if (c0 > 0) cost += 70 * N * H / (int64_t{8192} * 4096);
  }
  return cost;
}

// budget: bytes the plan may use (0 = the larger of N*V*4/16 and kBudgetFloor).
// Returns FLCE_OK or an error.
int make_plan(Plan* out, int64_t N, int64_t H, int64_t V, bool grads, const flce_opts& o,
              size_t budget) {
  Plan p;
  p.N = N;
  p.H = H;
  p.V = V;
  p.dtype = o.dtype;
  p.elt = (o.dtype == FLCE_FP32) ? 4 : 2;
  p.grads = grads;
  p.num_vblk = (V + BN - 1) / BN;
  p.cgrid = combine_grid(N);
  p.Np = (N + 3) / 4 * 4;
  const size_t fixed = fixed_bytes(p);
  if (grads && N > 0) {
    const int64_t vpad = p.num_vblk * BN;
    int64_t Vc;
    if (o.vocab_chunk > 0) {
      if (o.vocab_chunk % BN != 0) {
        set_error("vocab_chunk must be a positive multiple of %d", BN);
        return FLCE_ERR_ARG;
      }
      Vc = o.vocab_chunk;
    } else {
      if (budget == 0) {
        budget = static_cast<size_t>(N) * static_cast<size_t>(V) * 4 / 16;
        if (budget < kBudgetFloor) budget = kBudgetFloor;
      }
      size_t per_col = static_cast<size_t>(N) * p.elt;  // G chunk column
      if (p.dtype == FLCE_FP32)                            // + G^T and W^T columns
        per_col += static_cast<size_t>(p.Np) * 4 + static_cast<size_t>(H) * 4;
      const size_t avail = budget > fixed ? budget - fixed : 0;
      int64_t vmax = static_cast<int64_t>(avail / per_col) / BN * BN;
      // Narrower chunks cost more than they save: below kMinChunk columns the
      // dW GEMM has too few tiles to fill the GPU, so the budget is exceeded
      // rather than going below it.
      if (vmax < kMinChunk) vmax = kMinChunk;
      if (vmax > vpad) vmax = vpad;
      // Among the widths the budget allows, the one with the least estimated
      // time (ties: the widest, i.e. the fewest launches).
      const bool pair = (p.dtype == FLCE_BF16);
      Vc = vmax;
      int64_t best = chunk_loop_cost(N, H, V, vmax, p.elt, pair);
      for (int64_t w = vmax - BN; w >= kMinChunk; w -= BN) {
        const int64_t cst = chunk_loop_cost(N, H, V, w, p.elt, pair);
        if (cst < best) {
          best = cst;
          Vc = w;
        }
      }
    }
    if (Vc > vpad) Vc = vpad;
    p.Vc = Vc;
    p.num_chunks = (V + Vc - 1) / Vc;
    size_t o = fixed + align_up(static_cast<size_t>(N) * static_cast<size_t>(Vc) * p.elt, 256);
    p.off_gt = o;
    p.off_wt = o;
    if (p.dtype == FLCE_FP32) {
      o += align_up(static_cast<size_t>(Vc) * static_cast<size_t>(p.Np) * 4, 256);
      p.off_wt = o;
      o += align_up(static_cast<size_t>(H) * static_cast<size_t>(Vc) * 4, 256);
    }
    p.total = o;
  } else {
    p.total = fixed;
  }
  *out = p;
  return FLCE_OK;
}

int check_args(const void* X, const void* W, const int64_t* target, int64_t N, int64_t H,
               int64_t V, const flce_opts& o) {
  if (N < 0 || H <= 0 || V <= 0) {
    set_error("sizes must satisfy N >= 0, H > 0, V > 0 (got N=%lld H=%lld V=%lld)",
              static_cast<long long>(N), static_cast<long long>(H), static_cast<long long>(V));
    return FLCE_ERR_ARG;
  }
  if (o.dtype != FLCE_BF16 && o.dtype != FLCE_FP32) {
    set_error("unknown dtype %d", o.dtype);
    return FLCE_ERR_ARG;
  }
  if (N > (int64_t{1} << 31) - BM || V > (int64_t{1} << 31) - BN || H > (int64_t{1} << 24)) {
    set_error("size too large (N < 2^31, V < 2^31, H <= 2^24)");
    return FLCE_ERR_ARG;
  }
  if (!W || (N > 0 && (!X || !target))) {
    set_error("null input pointer");
    return FLCE_ERR_ARG;
  }
  const int elt = (o.dtype == FLCE_FP32) ? 4 : 2;
  if ((H * elt) % 16 != 0) {
    set_error("H * sizeof(element) = %lld is not a multiple of 16 bytes",
              static_cast<long long>(H * elt));
    return FLCE_ERR_ALIGN;
  }
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W)) & 15u) {
    set_error("X and W must be 16-byte aligned");
    return FLCE_ERR_ALIGN;
  }
  if (o.grad_scale != o.grad_scale) {
    set_error("grad_scale is NaN");
    return FLCE_ERR_ARG;
  }
  return FLCE_OK;
}

struct Tracer {
  const flce_opts& o;
  cudaStream_t s;
  int32_t n = 0;
  Tracer(const flce_opts& opts, cudaStream_t st) : o(opts), s(st) {}
  int start() {
    if (!o.trace_events || o.trace_capacity < 1) return FLCE_OK;
    FLCE_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(o.trace_events[0]), s));
    n = 1;
    return FLCE_OK;
  }
  int after(int kind) {
    if (!o.trace_events || n == 0 || n >= o.trace_capacity) return FLCE_OK;
    FLCE_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(o.trace_events[n]), s));
    if (o.trace_kinds) o.trace_kinds[n - 1] = kind;
    ++n;
    return FLCE_OK;
  }
  void finish() {
    if (o.trace_count) *o.trace_count = n;
  }
};

int grid_for(int64_t tiles, int sms) {
  return static_cast<int>(tiles < sms ? tiles : sms);
}

// Copies of the host-buffer entry that overlap the path: W arrives in pieces
// on a copy stream (pass 1 runs piece by piece as they land), and each chunk's
// dW rows go back to the host as soon as their GEMM is done.
struct HostOverlap {
  cudaStream_t copy;
  int32_t n_w_pieces;
  int64_t w_piece_tiles;        // vocabulary tiles of BN rows per piece
  const cudaEvent_t* w_ready;   // [n_w_pieces], recorded on `copy`
  float* dW_host;
  const cudaEvent_t* chunk_done;  // [num_chunks]
  cudaEvent_t copies_done;
};

// Rows of X that pass 1 keeps in L2 at a time (its M band), in bytes.
constexpr size_t kPass1BandBytes = size_t{32} << 20;
// dW walks H fastest inside bands of 8 H blocks: a wave of 76 pair tiles
// then covers about 9.5 vocabulary blocks x 8 H blocks of the output, and
// reads 9.5 slabs of G_c and half of X instead of 4.75 slabs and all of X.
// At 8192 x 4096, chunk 4864: 358 -> 294 MB read per launch; same-box A/B
// Llama-3 head +0.7 to +1.2% per call, Qwen2 head +0.6%, long context +1.0%.
constexpr int32_t kDwHBand = 8;

// The whole path on device pointers.  `ws` holds at least plan.total bytes.
int run_path(const Plan& P, const DeviceInfo& D, const void* X, const void* W,
             const int64_t* target, int64_t ignore_index, void* dX, float* dW, uint8_t* ws,
             const flce_opts& o, cudaStream_t s, const HostOverlap* ov = nullptr) {
  const int64_t N = P.N, H = P.H, V = P.V;
  const int elt = P.elt;
  const bool bf16 = (P.dtype == FLCE_BF16);
  const CUtensorMapDataType dt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const int KE = 128 / elt;  // K elements per 128-byte stage
  const int64_t MB = bf16 ? 2 * BM : BM;  // rows of one tile (bf16: a CTA pair)
  const uint32_t BR = bf16 ? BN / 2 : BN;  // rows of B one CTA stages (K-major box height)
  const int units = bf16 ? D.units_bf16 : D.units_fp32;
  Scalars* sc = reinterpret_cast<Scalars*>(ws + P.off_sc);
  float* lse2 = reinterpret_cast<float*>(ws + P.off_lse2);
  float* st = reinterpret_cast<float*>(ws + P.off_st);
  float* partial = reinterpret_cast<float*>(ws + P.off_partial);
  const Targets tg{target, o.target_is_int32 != 0 ? 1 : 0};
  int rc;
  Tracer tr(o, s);

  FLCE_CUDA(cudaMemsetAsync(sc, 0, sizeof(Scalars), s));
  if ((rc = tr.start())) return rc;

  // ---- pass 1 and combine
  if (N > 0) {
    CUtensorMap mX, mW;
    if ((rc = make_map(&mX, X, dt, elt, H, N, H * elt, KE, BM, "X (K-major)"))) return rc;
    if ((rc = make_map(&mW, W, dt, elt, H, V, H * elt, KE, BR, "W (K-major)"))) return rc;
    // one launch over the whole vocabulary, or one per uploaded piece of W
    const int64_t piece = ov ? ov->w_piece_tiles : P.num_vblk;
    for (int64_t t0 = 0, pi = 0; t0 < P.num_vblk; t0 += piece, ++pi) {
      const int64_t nt = (P.num_vblk - t0) < piece ? (P.num_vblk - t0) : piece;
      if (ov) FLCE_CUDA(cudaStreamWaitEvent(s, ov->w_ready[pi], 0));
      GemmGrid g{};
      g.num_m_blk = static_cast<int32_t>((N + MB - 1) / MB);
      g.num_n_blk = static_cast<int32_t>(nt);
      g.num_k_blk = static_cast<int32_t>((H + KE - 1) / KE);
      g.b_mn_off = static_cast<int32_t>(t0 * BN);
      g.status = &sc->status;
      // M fastest in bands of about 32 MiB of X rows: one band of X stays in
      // L2 while W streams through once per band (16 M blocks at H = 4096).
      // Same-box A/B against no bands: Llama-3 head -0.9%, Qwen2 head -3.6%,
      // long context -4% per call; 48 MiB bands measured the same.
      g.m_band = static_cast<int32_t>(kPass1BandBytes / (static_cast<size_t>(MB) * H * elt) > 0
                                          ? kPass1BandBytes / (static_cast<size_t>(MB) * H * elt)
                                          : 1);
      RowLseParams rp{tg, partial, st, N, V, static_cast<int32_t>(t0)};
      const int grid = grid_for(static_cast<int64_t>(g.num_m_blk) * g.num_n_blk, units);
      FLCE_CUDA(bf16 ? launch_logits_lse_bf16(mX, mW, g, rp, grid, s)
                     : launch_logits_lse_fp32(mX, mW, g, rp, grid, s));
      if ((rc = tr.after(FLCE_TRACE_LOGITS_LSE))) return rc;
    }
  }
  CombineParams cp{};
  cp.partial = partial;
  cp.num_vblk = static_cast<int32_t>(P.num_vblk);
  cp.st = st;
  cp.target = tg;
  cp.N = N;
  cp.V = V;
  cp.ignore_index = ignore_index;
  cp.lse2 = lse2;
  cp.lse_out = o.lse_out;
  cp.loss_rows_out = o.loss_rows_out;
  cp.blk_loss = reinterpret_cast<double*>(ws + P.off_blk_loss);
  cp.blk_cnt = reinterpret_cast<int64_t*>(ws + P.off_blk_cnt);
  cp.sc = sc;
  cp.grad_scale = o.grad_scale;
  cp.norm_count = o.norm_count;
  cp.loss_out = o.loss_dev;
  cp.nvalid_out = o.n_valid_dev;
  FLCE_CUDA(launch_combine(cp, s));
  if ((rc = tr.after(FLCE_TRACE_COMBINE))) return rc;

  // ---- pass 2 and the gradient GEMMs, chunk by chunk over the vocabulary
  if (P.grads) {
    if (N == 0) {
      FLCE_CUDA(cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * H * 4, s));
    } else {
      uint8_t* G = ws + P.off_G;
      float* dxacc = bf16 ? reinterpret_cast<float*>(ws + P.off_dxacc) : static_cast<float*>(dX);
      const int64_t Vc = P.Vc, Np = P.Np;
      float* Xt = reinterpret_cast<float*>(ws + P.off_xt);
      float* Gt = reinterpret_cast<float*>(ws + P.off_gt);
      float* Wt = reinterpret_cast<float*>(ws + P.off_wt);
      // A/B maps of the dW GEMM (mA4, mB4) and of the dX GEMM (mA5, mB5)
      CUtensorMap mX_K, mW_K, mG_st, mA4, mB4, mA5, mB5, mdW, mdX;
      if ((rc = make_map(&mX_K, X, dt, elt, H, N, H * elt, KE, BM, "X (K-major)"))) return rc;
      if ((rc = make_map(&mW_K, W, dt, elt, H, V, H * elt, KE, BR, "W (K-major)"))) return rc;
      if ((rc = make_map(&mG_st, G, dt, elt, Vc, N, Vc * elt, KE, 32, "G store"))) return rc;
      if ((rc = make_map(&mA5, G, dt, elt, Vc, N, Vc * elt, KE, BM, "G (K-major)"))) return rc;
      if (bf16) {
        if ((rc = make_map(&mA4, G, dt, elt, Vc, N, Vc * elt, KE, KE, "G (MN-major)")))
          return rc;
        if ((rc = make_map(&mB4, X, dt, elt, H, N, H * elt, KE, KE, "X (MN-major)"))) return rc;
        if ((rc = make_map(&mB5, W, dt, elt, H, V, H * elt, KE, KE, "W (MN-major)"))) return rc;
      } else {
        if ((rc = make_map(&mA4, Gt, dt, 4, N, Vc, Np * 4, KE, BM, "G^T (K-major)"))) return rc;
        if ((rc = make_map(&mB4, Xt, dt, 4, N, H, Np * 4, KE, BN, "X^T (K-major)"))) return rc;
        if ((rc = make_map(&mB5, Wt, dt, 4, Vc, H, Vc * 4, KE, BN, "W^T chunk (K-major)")))
          return rc;
        FLCE_CUDA(launch_transpose_f32(static_cast<const float*>(X), N, H, H, Xt, Np, Np,
                                       D.sms, s));
      }
      if ((rc = make_map(&mdW, dW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, V, H * 4, 32, 32,
                         "dW store")))
        return rc;
      if ((rc = make_map(&mdX, dxacc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, N, H * 4, 32, 32,
                         "dX accumulator")))
        return rc;
      const int32_t m_tok = static_cast<int32_t>((N + MB - 1) / MB);
      const int32_t n_h = static_cast<int32_t>((H + BN - 1) / BN);
      for (int64_t c = 0; c < P.num_chunks; ++c) {
        const int64_t c0 = c * Vc;
        const int64_t vc = (V - c0) < Vc ? (V - c0) : Vc;
        // pass 2: G_c
        {
          GemmGrid g{};
          g.num_m_blk = m_tok;
          g.num_n_blk = static_cast<int32_t>((vc + BN - 1) / BN);
          g.num_k_blk = static_cast<int32_t>((H + KE - 1) / KE);
          g.b_mn_off = static_cast<int32_t>(c0);
          g.status = &sc->status;
          // N fastest: the chunk's W rows (Vc x H, 40 MB at the Llama-3 head)
          // stay in L2 while X streams once (M fastest re-read X from DRAM:
          // 332 against 121 MB per launch at 8192 x 4096, Vc 4864)
          g.raster_n = 1;
          // operands are inputs: the loads start at once; the epilogue
          // waits for the previous launch before it overwrites G
          GradLogitsParams gp{tg, lse2, sc, N, V, ignore_index, c0};
          const int grid = grid_for(static_cast<int64_t>(g.num_m_blk) * g.num_n_blk, units);
          FLCE_CUDA(bf16 ? launch_logits_grad_bf16(mX_K, mW_K, mG_st, g, gp, grid, s)
                         : launch_logits_grad_fp32(mX_K, mW_K, mG_st, g, gp, grid, s));
          if ((rc = tr.after(FLCE_TRACE_LOGITS_GRAD))) return rc;
        }
        if (!bf16) {
          FLCE_CUDA(launch_transpose_f32(reinterpret_cast<const float*>(G), N, Vc, Vc, Gt, Np,
                                         Np, D.sms, s));
          FLCE_CUDA(launch_transpose_f32(static_cast<const float*>(W) + c0 * H, vc, H, H, Wt,
                                         Vc, Vc, D.sms, s));
        }
        // dW[c0 : c0+vc] = G_c^T X
        {
          GemmGrid g{};
          g.num_m_blk = static_cast<int32_t>((vc + MB - 1) / MB);
          g.num_n_blk = n_h;
          g.num_k_blk = static_cast<int32_t>((N + KE - 1) / KE);
          g.status = &sc->status;
          g.raster_n = 1;  // a slab of G_c rows with all of X stays in L2
          g.n_band = kDwHBand;
          g.wait_operands = 1;  // G_c comes from the launch just before
          StoreParams sp{0, static_cast<int32_t>(c0), 0};
          const int grid = grid_for(static_cast<int64_t>(g.num_m_blk) * g.num_n_blk, units);
          FLCE_CUDA(bf16 ? launch_dw_bf16(mA4, mB4, mdW, g, sp, grid, s)
                         : launch_dw_fp32(mA4, mB4, mdW, g, sp, grid, s));
          if ((rc = tr.after(FLCE_TRACE_DW))) return rc;
          if (ov) {  // these dW rows are final: send them to the host now
            FLCE_CUDA(cudaEventRecord(ov->chunk_done[c], s));
            FLCE_CUDA(cudaStreamWaitEvent(ov->copy, ov->chunk_done[c], 0));
            FLCE_CUDA(cudaMemcpyAsync(ov->dW_host + c0 * H, dW + c0 * H,
                                      static_cast<size_t>(vc) * H * 4, cudaMemcpyDeviceToHost,
                                      ov->copy));
          }
        }
        // dX_acc (+)= G_c W[c0 : c0+vc]
        {
          GemmGrid g{};
          g.num_m_blk = m_tok;
          g.num_n_blk = n_h;
          g.num_k_blk = static_cast<int32_t>((vc + KE - 1) / KE);
          g.b_k_off = bf16 ? static_cast<int32_t>(c0) : 0;
          g.raster_n = 1;  // a slab of G_c rows with all of W[c] stays in L2
          g.status = &sc->status;
          // G_c comes from two launches back (the dW launch is in between),
          // so the operand loads start at once
          StoreParams sp{0, 0, c > 0 ? 1 : 0};
          const int grid = grid_for(static_cast<int64_t>(g.num_m_blk) * g.num_n_blk, units);
          FLCE_CUDA(bf16 ? launch_dx_bf16(mA5, mB5, mdX, g, sp, grid, s)
                         : launch_dx_fp32(mA5, mB5, mdX, g, sp, grid, s));
          if ((rc = tr.after(FLCE_TRACE_DX))) return rc;
        }
      }
      if (bf16) {
        FLCE_CUDA(launch_convert_bf16(dxacc, dX, N * H, D.sms, s));
        if ((rc = tr.after(FLCE_TRACE_CONVERT))) return rc;
      }
    }
  }
  if (ov && N > 0) {  // the compute stream continues only once dW is home
    FLCE_CUDA(cudaEventRecord(ov->copies_done, ov->copy));
    FLCE_CUDA(cudaStreamWaitEvent(s, ov->copies_done, 0));
  }
  if (o.status_dev) FLCE_CUDA(launch_status_code(sc, o.status_dev, s));
  tr.finish();
  return FLCE_OK;
}

int status_from_bits(int32_t bits) {
  if (bits & FLCE_DEV_TIMEOUT) {
    set_error("a bounded wait inside a kernel expired");
    return FLCE_ERR_TIMEOUT;
  }
  if (bits & FLCE_DEV_TARGET) {
    set_error("a target is outside [0, V) and is not the ignore index");
    return FLCE_ERR_TARGET;
  }
  return FLCE_OK;
}

int entry(const void* X, const void* W, const int64_t* target, int64_t N, int64_t H, int64_t V,
          int64_t ignore_index, float* loss_host, void* dX, float* dW, const flce_opts* opts_in,
          bool grads, const HostOverlap* ov = nullptr) {
  g_last_error[0] = 0;
  flce_opts o;
  flce_opts_init(&o);
  if (opts_in) o = *opts_in;
  int rc = check_args(X, W, target, N, H, V, o);
  if (rc) return rc;
  if (grads) {
    if (!dW || (N > 0 && !dX)) {
      set_error("null gradient pointer");
      return FLCE_ERR_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(dX) | reinterpret_cast<uintptr_t>(dW)) & 15u) {
      set_error("dX and dW must be 16-byte aligned");
      return FLCE_ERR_ALIGN;
    }
  }
  const bool sync = o.sync != 0 || loss_host != nullptr;
  DeviceInfo D;
  if ((rc = device_info(o.dtype, &D))) return rc;

  Plan P;
  if ((rc = make_plan(&P, N, H, V, grads, o, o.workspace ? o.workspace_bytes : o.workspace_budget)))
    return rc;
  if (o.workspace && o.workspace_bytes < P.total) {
    set_error("workspace of %zu bytes is smaller than the %zu bytes this call needs",
              o.workspace_bytes, P.total);
    return FLCE_ERR_WORKSPACE;
  }
  if (o.workspace && (reinterpret_cast<uintptr_t>(o.workspace) & 255u)) {
    set_error("workspace must be 256-byte aligned");
    return FLCE_ERR_ALIGN;
  }
  if (o.workspace_used) *o.workspace_used = P.total;
  if (o.vocab_chunk_used) *o.vocab_chunk_used = P.Vc;

  cudaStream_t s = static_cast<cudaStream_t>(o.stream);
  uint8_t* ws = static_cast<uint8_t*>(o.workspace);
  bool owned = false;
  if (!ws) {
    void* p = nullptr;
    if ((rc = pool_alloc(&p, P.total, s))) return rc;
    ws = static_cast<uint8_t*>(p);
    owned = true;
  }
  rc = run_path(P, D, X, W, target, ignore_index, dX, dW, ws, o, s, ov);
  Scalars host_sc{};
  if (rc == FLCE_OK && sync) {
    cudaError_t e = cudaMemcpyAsync(&host_sc, ws + P.off_sc, sizeof(Scalars),
                                    cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemcpyAsync(scalars)");
  }
  if (owned) {
    cudaError_t e = cudaFreeAsync(ws, s);
    if (e != cudaSuccess && rc == FLCE_OK) rc = cuda_fail(e, "cudaFreeAsync(workspace)");
  }
  if (rc != FLCE_OK) return rc;
  if (sync) {
    FLCE_CUDA(cudaStreamSynchronize(s));
    if ((rc = status_from_bits(host_sc.status))) return rc;
    if (loss_host) *loss_host = host_sc.loss;
  }
  return FLCE_OK;
}

// Cross-entropy on materialised logits: count, rows, combine.
int ce_entry(const void* logits, const int64_t* target, int64_t N, int64_t V,
             int64_t ignore_index, float* loss_host, void* dlogits, const flce_opts* opts_in) {
  g_last_error[0] = 0;
  flce_opts o;
  flce_opts_init(&o);
  if (opts_in) o = *opts_in;
  if (N < 0 || V <= 0 || (N > 0 && (!logits || !target))) {
    set_error("bad arguments (need N >= 0, V > 0 and non-null logits and target)");
    return FLCE_ERR_ARG;
  }
  if (o.dtype != FLCE_BF16 && o.dtype != FLCE_FP32) {
    set_error("unknown dtype %d", o.dtype);
    return FLCE_ERR_ARG;
  }
  if (N > (int64_t{1} << 31) || V > (int64_t{1} << 31)) {
    set_error("size too large (N, V <= 2^31)");
    return FLCE_ERR_ARG;
  }
  const int elt = (o.dtype == FLCE_FP32) ? 4 : 2;
  const Targets tg{target, o.target_is_int32 != 0 ? 1 : 0};
  DeviceInfo D;
  int rc = device_info(o.dtype, &D);
  if (rc) return rc;
  const bool sync = o.sync != 0 || loss_host != nullptr;
  const int cgrid = combine_grid(N);
  size_t off = 0;
  const size_t off_sc = off;
  off += align_up(sizeof(Scalars), 256);
  const size_t off_bl = off;
  off += align_up(static_cast<size_t>(cgrid) * 8, 256);
  const size_t off_bc = off;
  off += align_up(static_cast<size_t>(cgrid) * 8, 256);
  const size_t off_lse2 = off;
  off += align_up(static_cast<size_t>(N) * 4, 256);
  const size_t off_st = off;
  off += align_up(static_cast<size_t>(N) * 4, 256);
  const size_t off_part = off;
  off += align_up(static_cast<size_t>(N) * 4, 256);
  const size_t total = off;
  if (o.workspace_used) *o.workspace_used = total;
  if (o.workspace && o.workspace_bytes < total) {
    set_error("workspace of %zu bytes is smaller than the %zu bytes this call needs",
              o.workspace_bytes, total);
    return FLCE_ERR_WORKSPACE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(o.stream);
  uint8_t* ws = static_cast<uint8_t*>(o.workspace);
  bool owned = false;
  if (!ws) {
    void* pws = nullptr;
    if ((rc = pool_alloc(&pws, total, s))) return rc;
    ws = static_cast<uint8_t*>(pws);
    owned = true;
  }
  Scalars* sc = reinterpret_cast<Scalars*>(ws + off_sc);
  Tracer tr(o, s);
  cudaError_t e = cudaMemsetAsync(sc, 0, sizeof(Scalars), s);
  if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemsetAsync(scalars)");
  if (rc == FLCE_OK) rc = tr.start();
  if (rc == FLCE_OK && N > 0) {
    e = launch_ce_count(tg, N, V, ignore_index, sc, D.sms, s);
    if (e != cudaSuccess) rc = cuda_fail(e, "ce_count");
    if (rc == FLCE_OK) rc = tr.after(FLCE_TRACE_CE_COUNT);
  }
  if (rc == FLCE_OK && N > 0) {
    CeRowsParams cp{};
    cp.logits = logits;
    cp.dlogits = dlogits;
    cp.target = tg;
    cp.N = N;
    cp.V = V;
    cp.ignore_index = ignore_index;
    cp.sc = sc;
    cp.grad_scale = o.grad_scale;
    cp.norm_count = o.norm_count;
    cp.partial = reinterpret_cast<float*>(ws + off_part);
    cp.st = reinterpret_cast<float*>(ws + off_st);
    cp.vectorized = ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(dlogits)) &
                     15u) == 0 &&
                    (V * elt) % 16 == 0 && (V * elt) / 16 < (int64_t{1} << 30);
    e = launch_ce_rows(cp, elt, D.sms, s);
    if (e != cudaSuccess) rc = cuda_fail(e, "ce_rows");
    if (rc == FLCE_OK) rc = tr.after(FLCE_TRACE_CE_ROWS);
  }
  if (rc == FLCE_OK) {
    CombineParams cp{};
    cp.partial = reinterpret_cast<float*>(ws + off_part);
    cp.num_vblk = 1;
    cp.st = reinterpret_cast<float*>(ws + off_st);
    cp.target = tg;
    cp.N = N;
    cp.V = V;
    cp.ignore_index = ignore_index;
    cp.lse2 = reinterpret_cast<float*>(ws + off_lse2);
    cp.lse_out = o.lse_out;
    cp.loss_rows_out = o.loss_rows_out;
    cp.blk_loss = reinterpret_cast<double*>(ws + off_bl);
    cp.blk_cnt = reinterpret_cast<int64_t*>(ws + off_bc);
    cp.sc = sc;
    cp.grad_scale = o.grad_scale;
    cp.norm_count = o.norm_count;
    cp.loss_out = o.loss_dev;
    cp.nvalid_out = o.n_valid_dev;
    e = launch_combine(cp, s);
    if (e != cudaSuccess) rc = cuda_fail(e, "combine");
    if (rc == FLCE_OK) rc = tr.after(FLCE_TRACE_COMBINE);
  }
  if (rc == FLCE_OK && o.status_dev) {
    e = launch_status_code(sc, o.status_dev, s);
    if (e != cudaSuccess) rc = cuda_fail(e, "status");
  }
  tr.finish();
  Scalars host_sc{};
  if (rc == FLCE_OK && sync) {
    e = cudaMemcpyAsync(&host_sc, sc, sizeof(Scalars), cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemcpyAsync(scalars)");
  }
  if (owned) {
    e = cudaFreeAsync(ws, s);
    if (e != cudaSuccess && rc == FLCE_OK) rc = cuda_fail(e, "cudaFreeAsync(workspace)");
  }
  if (rc != FLCE_OK) return rc;
  if (sync) {
    FLCE_CUDA(cudaStreamSynchronize(s));
    if ((rc = status_from_bits(host_sc.status))) return rc;
    if (loss_host) *loss_host = host_sc.loss;
  }
  return FLCE_OK;
}

}  // namespace
}  // namespace flce

// ------------------------------------------------ allocation-free loss entry
// Scratch of flce_fwd_noalloc(): a fixed device array owned by this library.
// Every device on which the library runs a kernel holds it until the process
// exits.  Host code must not pass `g_noalloc_scratch` itself to a kernel (on
// the host that name is only a stand-in for the device symbol); its device
// address comes from cudaGetSymbolAddress() below.
constexpr size_t kNoAllocScratchBytes = size_t{32} << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace flce {
namespace {

void* g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mutex;

// Device address of the scratch array on the current device, looked up once
// per device (the lookup may load the library's kernels onto the device).
int noalloc_scratch(void** out) {
  int dev = 0;
  FLCE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal %d out of range", dev);
    return FLCE_ERR_ARG;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return FLCE_OK;
}

}  // namespace
}  // namespace flce

using namespace flce;

extern "C" {

void flce_opts_init(flce_opts* o) {
  if (!o) return;
  std::memset(o, 0, sizeof *o);
  o->dtype = FLCE_BF16;
  o->sync = 1;
  o->grad_scale = 1.0f;
}

int flce_fwd_bwd(const void* X, const void* W, const int64_t* target, int64_t N, int64_t H,
                 int64_t V, int64_t ignore_index, float* loss, void* dX, float* dW) {
  if (!loss) {
    set_error("loss pointer is null");
    return FLCE_ERR_ARG;
  }
  return entry(X, W, target, N, H, V, ignore_index, loss, dX, dW, nullptr, true);
}

int flce_fwd_bwd_ex(const void* X, const void* W, const int64_t* target, int64_t N, int64_t H,
                    int64_t V, int64_t ignore_index, float* loss, void* dX, float* dW,
                    const flce_opts* opts) {
  return entry(X, W, target, N, H, V, ignore_index, loss, dX, dW, opts, true);
}

int flce_fwd(const void* X, const void* W, const int64_t* target, int64_t N, int64_t H, int64_t V,
             int64_t ignore_index, float* loss, const flce_opts* opts) {
  return entry(X, W, target, N, H, V, ignore_index, loss, nullptr, nullptr, opts, false);
}

int flce_fwd_bwd_host(const void* X_host, const void* W_host, const int64_t* target_host,
                      int64_t N, int64_t H, int64_t V, int64_t ignore_index, float* loss,
                      void* dX_host, float* dW_host, const flce_opts* opts_in) {
  g_last_error[0] = 0;
  flce_opts o;
  flce_opts_init(&o);
  if (opts_in) o = *opts_in;
  if (!loss || !dW_host || !W_host || (N > 0 && (!X_host || !target_host || !dX_host))) {
    set_error("null host pointer");
    return FLCE_ERR_ARG;
  }
  if (N < 0 || H <= 0 || V <= 0 || (o.dtype != FLCE_BF16 && o.dtype != FLCE_FP32)) {
    set_error("bad sizes or dtype");
    return FLCE_ERR_ARG;
  }
  Plan P;
  int rc = make_plan(&P, N, H, V, true, o, o.workspace_budget);
  if (rc) return rc;
  const size_t elt = (o.dtype == FLCE_FP32) ? 4 : 2;
  const size_t bx = static_cast<size_t>(N) * H * elt, bw = static_cast<size_t>(V) * H * elt,
               bt = static_cast<size_t>(N) * (o.target_is_int32 ? 4 : 8),
               bdw = static_cast<size_t>(V) * H * 4;
  cudaStream_t s = static_cast<cudaStream_t>(o.stream);
  const size_t ox = 0, ow = align_up(ox + bx, 256), ot = align_up(ow + bw, 256),
               odx = align_up(ot + bt, 256), odw = align_up(odx + bx, 256),
               osc = align_up(odw + bdw, 256), total = osc + 256;
  // W goes up in pieces of whole vocabulary tiles, pass 1 following them
  constexpr int kPieces = 8;
  const int64_t piece_tiles = (P.num_vblk + kPieces - 1) / kPieces;
  const int n_pieces = static_cast<int>((P.num_vblk + piece_tiles - 1) / piece_tiles);
  const int n_chunks = static_cast<int>(P.num_chunks);
  void* buf = nullptr;
  if ((rc = pool_alloc(&buf, total, s))) return rc;
  uint8_t* b = static_cast<uint8_t*>(buf);
  float* loss_dev = reinterpret_cast<float*>(b + osc);
  int32_t* status_dev = reinterpret_cast<int32_t*>(b + osc + 16);
  cudaStream_t cs = nullptr;
  const int n_events = n_pieces + n_chunks + 2;
  cudaEvent_t* ev = new cudaEvent_t[n_events]();
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  for (int i = 0; e == cudaSuccess && i < n_events; ++i)
    e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
  cudaEvent_t* w_ready = ev;
  cudaEvent_t* chunk_done = ev + n_pieces;
  cudaEvent_t alloc_ready = ev[n_events - 2], copies_done = ev[n_events - 1];
  if (e == cudaSuccess) e = cudaEventRecord(alloc_ready, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, alloc_ready, 0);
  if (e == cudaSuccess && bx) e = cudaMemcpyAsync(b + ox, X_host, bx, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && bt)
    e = cudaMemcpyAsync(b + ot, target_host, bt, cudaMemcpyHostToDevice, s);
  for (int p = 0; e == cudaSuccess && p < n_pieces; ++p) {
    const int64_t r0 = p * piece_tiles * BN;
    const int64_t r1 = (r0 + piece_tiles * BN) < V ? (r0 + piece_tiles * BN) : V;
    const size_t off = static_cast<size_t>(r0) * H * elt, len = static_cast<size_t>(r1 - r0) * H * elt;
    e = cudaMemcpyAsync(b + ow + off, static_cast<const uint8_t*>(W_host) + off, len,
                        cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaEventRecord(w_ready[p], cs);
  }
  if (e != cudaSuccess) rc = cuda_fail(e, "host-buffer staging");
  if (rc == FLCE_OK) {
    HostOverlap ov{cs, n_pieces, piece_tiles, w_ready, dW_host, chunk_done, copies_done};
    if (N == 0) {  // no pass 1 waits on the pieces: order the stream after them
      e = cudaEventRecord(copies_done, cs);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, copies_done, 0);
      if (e != cudaSuccess) rc = cuda_fail(e, "host-buffer staging");
    }
    flce_opts io = o;
    io.sync = 0;
    io.loss_dev = loss_dev;
    io.status_dev = status_dev;
    if (rc == FLCE_OK)
      rc = entry(b + ox, b + ow, reinterpret_cast<const int64_t*>(b + ot), N, H, V, ignore_index,
                 nullptr, b + odx, reinterpret_cast<float*>(b + odw), &io, true,
                 N > 0 ? &ov : nullptr);
  }
  float h_loss = 0.f;
  int32_t h_status = 0;
  if (rc == FLCE_OK) {
    e = cudaSuccess;
    if (N == 0) e = cudaMemcpyAsync(dW_host, b + odw, bdw, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && bx) e = cudaMemcpyAsync(dX_host, b + odx, bx, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h_loss, loss_dev, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h_status, status_dev, 4, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemcpyAsync(D2H)");
  }
  e = cudaFreeAsync(buf, s);
  if (e != cudaSuccess && rc == FLCE_OK) rc = cuda_fail(e, "cudaFreeAsync");
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess && rc == FLCE_OK) rc = cuda_fail(e, "cudaStreamSynchronize");
  if (cs) {
    cudaStreamSynchronize(cs);
    cudaStreamDestroy(cs);
  }
  for (int i = 0; i < n_events; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  delete[] ev;
  if (rc != FLCE_OK) return rc;
  if (h_status == FLCE_ERR_TIMEOUT || h_status == FLCE_ERR_TARGET) {
    set_error("%s", flce_status_str(h_status));
    return h_status;
  }
  *loss = h_loss;
  return FLCE_OK;
}

size_t flce_workspace_bytes(int64_t N, int64_t H, int64_t V, int with_grads,
                            const flce_opts* opts_in) {
  flce_opts o;
  flce_opts_init(&o);
  if (opts_in) o = *opts_in;
  if (N < 0 || H <= 0 || V <= 0) return 0;
  Plan P;
  if (make_plan(&P, N, H, V, with_grads != 0, o, o.workspace_budget) != FLCE_OK) return 0;
  return P.total;
}

const char* flce_status_str(int s) {
  switch (s) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_ARG: return "invalid argument";
    case FLCE_ERR_ALIGN: return "misaligned pointer or row pitch";
    case FLCE_ERR_ARCH: return "device is not compute capability 10.3";
    case FLCE_ERR_TARGET: return "target outside [0, V) that is not the ignore index";
    case FLCE_ERR_WORKSPACE: return "workspace too small";
    case FLCE_ERR_CUDA: return "CUDA error";
    case FLCE_ERR_TIMEOUT: return "bounded wait expired inside a kernel";
    default: return "unknown status";
  }
}

const char* flce_last_error(void) { return g_last_error; }

int flce_version(void) { return FLCE_VERSION; }

size_t flce_opts_sizeof(void) { return sizeof(flce_opts); }

int flce_ce_fwd_bwd(const void* logits, const int64_t* target, int64_t N, int64_t V,
                    int64_t ignore_index, float* loss, void* dlogits, const flce_opts* opts) {
  return ce_entry(logits, target, N, V, ignore_index, loss, dlogits, opts);
}

int flce_selftest_wait_expiry(int64_t limit_ns) {
  g_last_error[0] = 0;
  if (limit_ns <= 0 || limit_ns > 2000000000) {
    set_error("limit_ns must be in (0, 2e9]");
    return FLCE_ERR_ARG;
  }
  DeviceInfo D;
  int rc = device_info(FLCE_BF16, &D);
  if (rc) return rc;
  void* p = nullptr;
  FLCE_CUDA(cudaMalloc(&p, sizeof(Scalars)));
  Scalars* sc = static_cast<Scalars*>(p);
  Scalars h{};
  cudaError_t e = cudaMemset(sc, 0, sizeof(Scalars));
  if (e == cudaSuccess) e = launch_wait_expiry(sc, static_cast<uint64_t>(limit_ns), nullptr);
  if (e == cudaSuccess) e = cudaMemcpy(&h, sc, sizeof(Scalars), cudaMemcpyDeviceToHost);
  cudaFree(p);
  if (e != cudaSuccess) return cuda_fail(e, "wait-expiry self-test");
  return status_from_bits(h.status);
}

int flce_scale_convert(const void* src, int32_t src_dtype, void* dst, int32_t dst_dtype,
                       int64_t n, const float* scale_dev, void* stream) {
  g_last_error[0] = 0;
  const bool ok_types = (src_dtype == FLCE_BF16 || src_dtype == FLCE_FP32) &&
                        (dst_dtype == FLCE_BF16 || dst_dtype == FLCE_FP32);
  if (n < 0 || !ok_types || (n > 0 && (!src || !dst))) {
    set_error("flce_scale_convert: bad arguments (n >= 0, known types, non-null buffers)");
    return FLCE_ERR_ARG;
  }
  const size_t se = src_dtype == FLCE_FP32 ? 4 : 2, de = dst_dtype == FLCE_FP32 ? 4 : 2;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  const uintptr_t s1 = s0 + static_cast<size_t>(n) * se, d1 = d0 + static_cast<size_t>(n) * de;
  const bool in_place = (s0 == d0 && se == de);
  if (n > 0 && !in_place && s0 < d1 && d0 < s1) {
    set_error("flce_scale_convert: dst overlaps src (only an exact in-place call of one type "
              "is allowed)");
    return FLCE_ERR_ARG;
  }
  DeviceInfo D;
  int rc = device_info(FLCE_BF16, &D);
  if (rc) return rc;
  FLCE_CUDA(launch_scale_convert(src, static_cast<int>(se), dst, static_cast<int>(de), n,
                                 scale_dev, D.sms, static_cast<cudaStream_t>(stream)));
  return FLCE_OK;
}

int flce_fwd_noalloc(const void* X, const void* W, const int64_t* target, int64_t N, int64_t H,
                     int64_t V, int64_t ignore_index, int32_t dtype, float* loss_dev,
                     float* lse_out, int64_t* n_valid_dev, int32_t* status_dev, void* stream) {
  g_last_error[0] = 0;
  flce_opts o;
  flce_opts_init(&o);
  o.dtype = dtype;
  o.sync = 0;
  o.stream = stream;
  o.loss_dev = loss_dev;
  o.lse_out = lse_out;
  o.n_valid_dev = n_valid_dev;
  o.status_dev = status_dev;
  if (!loss_dev) {
    set_error("loss_dev is null");
    return FLCE_ERR_ARG;
  }
  int rc = check_args(X, W, target, N, H, V, o);
  if (rc) return rc;
  DeviceInfo D;
  if ((rc = device_info(o.dtype, &D))) return rc;
  Plan P;
  if ((rc = make_plan(&P, N, H, V, false, o, 0))) return rc;
  if (P.total > kNoAllocScratchBytes) {
    set_error("flce_fwd_noalloc: this problem needs %zu bytes of scratch, more than the %zu "
              "bytes of the library's static scratch array",
              P.total, kNoAllocScratchBytes);
    return FLCE_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  if ((rc = noalloc_scratch(&ws))) return rc;
  o.workspace = ws;
  o.workspace_bytes = kNoAllocScratchBytes;
  // run_path clears the words that must start at zero (status, the combine's
  // ticket) on the stream before its first kernel; every other scratch byte
  // is written before it is read.
  return run_path(P, D, X, W, target, ignore_index, nullptr, nullptr,
                  static_cast<uint8_t*>(ws), o, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
