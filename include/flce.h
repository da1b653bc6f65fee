/*
 * flce.h -- C ABI of libflce, a fused linear cross-entropy engine for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (Liger-Kernel project overview, "Método de API de Baixo
 * Nível": loss = loss_fn(weight, input, target) followed by loss.backward();
 * "Cálculo Preciso": forward and backward are exact, not approximations):
 *
 *   S       = X W^T                 X [N, H] tokens, W [V, H] LM-head weight
 *   lse_i   = log sum_j exp(S_ij)   (natural log)
 *   valid_i = (target_i != ignore_index),  n = sum_i valid_i
 *   loss    = (1/n) sum_{valid i} (lse_i - S_{i, target_i})
 *   G_ij    = valid_i (softmax(S_i)_j - [j == target_i]) * grad_scale / n
 *   dX      = G W   [N, H],   dW = G^T X   [V, H]
 *
 * The N x V logits are never written to device memory: the kernels recompute
 * logit tiles in tensor memory and process the vocabulary in chunks, so the
 * scratch space grows with a chunk width, not with N x V (the pages' "input
 * chunking" and "fusão de kernels", Liger Kernel paper summary, 方法详解, and
 * the overview's "Princípios Técnicos").
 *
 * Conventions shared by every entry point
 *   - X, W and dX are row-major and contiguous, element type opts->dtype
 *     (bf16 by default, or fp32 computed with tf32 tensor-core products);
 *     dW is fp32; target is int64 [N] (int32 [N] when opts->target_is_int32
 *     is set; the pointer is then read as int32_t*).  All of them are device
 *     pointers owned by the caller, except in flce_fwd_bwd_host().
 *   - X, W, dX and dW must be 16-byte aligned and H * sizeof(element) must be
 *     a multiple of 16 bytes; otherwise FLCE_ERR_ALIGN.
 *   - dX and dW are overwritten, never accumulated into.
 *   - When no row is valid (n == 0, including N == 0) the loss is 0 and both
 *     gradients are 0; the call succeeds.
 *   - A target outside [0, V) that is not ignore_index makes the call return
 *     FLCE_ERR_TARGET (synchronous calls) or sets that code in
 *     opts->status_dev (asynchronous calls); outputs are then unspecified.
 *   - Every kernel-side wait is bounded; an expired wait is reported as
 *     FLCE_ERR_TIMEOUT, never as a device trap.
 *   - The library needs a compute capability 10.3 device (FLCE_ERR_ARCH).
 *   - Calls are reentrant; the only process-wide state is a per-device cache
 *     of device attributes and kernel attributes, and one stream-ordered
 *     memory pool per device for the scratch the library allocates itself
 *     (it keeps freed scratch mapped for reuse until the process exits, so
 *     it holds at most the largest scratch of the calls made so far).
 *   - An asynchronous call (opts->sync == 0, host loss NULL, no trace events)
 *     makes only stream-ordered CUDA calls: scratch allocation and release,
 *     memsets and kernel launches.  It can therefore be captured into a CUDA
 *     graph (after one call outside the capture has set up the per-device
 *     state), and replays reproduce an eager call bit for bit.
 *   - Nothing throws across this boundary; every entry returns an int status.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FLCE_VERSION 2

#if defined(__GNUC__)
#define FLCE_API __attribute__((visibility("default")))
#else
#define FLCE_API
#endif

typedef enum flce_status {
  FLCE_OK = 0,
  FLCE_ERR_ARG = 1,       /* null pointer, negative or zero size, bad option */
  FLCE_ERR_ALIGN = 2,     /* pointer or row pitch not 16-byte aligned */
  FLCE_ERR_ARCH = 3,      /* device is not compute capability 10.3 */
  FLCE_ERR_TARGET = 4,    /* target outside [0, V) that is not ignore_index */
  FLCE_ERR_WORKSPACE = 5, /* caller workspace smaller than the minimum plan */
  FLCE_ERR_CUDA = 6,      /* CUDA runtime / driver error (see flce_last_error) */
  FLCE_ERR_TIMEOUT = 7    /* a bounded wait inside a kernel expired */
} flce_status;

typedef enum flce_dtype {
  FLCE_BF16 = 0, /* X, W, dX bfloat16; products on tensor cores, fp32 accumulate */
  FLCE_FP32 = 1  /* X, W, dX float32; tf32 tensor-core products, fp32 accumulate */
} flce_dtype;

/* Launch kinds reported by the optional per-launch trace. */
typedef enum flce_trace_kind {
  FLCE_TRACE_LOGITS_LSE = 1,   /* pass 1: logit tiles -> per-tile row statistics */
  FLCE_TRACE_COMBINE = 2,      /* row logsumexp, row loss, mean, n_valid */
  FLCE_TRACE_LOGITS_GRAD = 3,  /* pass 2: logit tiles -> G chunk */
  FLCE_TRACE_DW = 4,           /* dW[chunk] = G_chunk^T X */
  FLCE_TRACE_DX = 5,           /* dX += G_chunk W[chunk] */
  FLCE_TRACE_CONVERT = 6,      /* fp32 dX accumulator -> bf16 dX */
  FLCE_TRACE_CE_COUNT = 7,     /* cross-entropy on logits: valid-row count */
  FLCE_TRACE_CE_ROWS = 8       /* cross-entropy on logits: row statistics + gradient */
} flce_trace_kind;

/*
 * Options.  Initialise with flce_opts_init(); every field then has a usable
 * default.  Pointers marked "optional" may stay NULL.
 */
typedef struct flce_opts {
  int32_t dtype;            /* flce_dtype of X, W and dX (default FLCE_BF16) */
  int32_t sync;             /* 1: block until done and report kernel-side errors
                               (default 1); 0: asynchronous on `stream` */
  void* stream;             /* cudaStream_t to launch on (default NULL = legacy
                               default stream) */
  void* workspace;          /* optional device scratch; NULL = the library
                               allocates it stream-ordered and frees it before
                               returning (stream-ordered) */
  size_t workspace_bytes;   /* size of `workspace` */
  size_t workspace_budget;  /* planner budget when workspace == NULL; 0 = one
                               sixteenth of the N x V fp32 logits, but at
                               least 96 MiB */
  int64_t vocab_chunk;      /* vocabulary columns per chunk; 0 = planner;
                               otherwise a positive multiple of 256 */
  float grad_scale;         /* multiplies G, hence dX and dW (default 1) */
  int32_t target_is_int32;  /* 1: `target` points to int32 ids [N] instead of
                               int64 (default 0) */
  int64_t norm_count;       /* > 0: normalise by this count instead of the
                               local n (a data-parallel shard normalising by
                               the global count); the loss is then
                               sum(row losses) / norm_count */
  float* loss_dev;          /* optional device float: the loss */
  float* lse_out;           /* optional device float[N]: lse_i (natural log) */
  float* loss_rows_out;     /* optional device float[N]: lse_i - S_{i,t_i}, 0
                               for ignored rows */
  int64_t* n_valid_dev;     /* optional device int64: n */
  int32_t* status_dev;      /* optional device int32: flce_status of the
                               kernels (asynchronous error reporting) */
  size_t* workspace_used;   /* optional host size_t: scratch bytes used */
  int64_t* vocab_chunk_used;/* optional host int64: chunk width used */
  void** trace_events;      /* optional cudaEvent_t[trace_capacity]: event 0 is
                               recorded before the first launch and event k
                               after launch k */
  int32_t* trace_kinds;     /* optional int32[trace_capacity]: kind of launch k
                               at index k-1 */
  int32_t trace_capacity;
  int32_t* trace_count;     /* optional host int32: events recorded */
} flce_opts;

/* Fill *opts with defaults (dtype bf16, sync 1, grad_scale 1, rest 0/NULL). */
FLCE_API void flce_opts_init(flce_opts* opts);

/*
 * Loss and both gradients, synchronous, default stream, bf16 inputs.
 *   X [N, H] bf16, W [V, H] bf16, target [N] int64   (device, read only)
 *   loss  host float* (required): the mean loss
 *   dX [N, H] bf16 and dW [V, H] fp32 (device, written)
 * Argument order: input rows, LM-head weight, targets (the hidden-states-first
 * call of the Liger Kernel command sheet, 常用示例); the Python binding keeps
 * the overview's loss_fn(weight, input, target) order instead.
 */
FLCE_API int flce_fwd_bwd(const void* X, const void* W, const int64_t* target, int64_t N, int64_t H,
                 int64_t V, int64_t ignore_index, float* loss, void* dX, float* dW);

/*
 * As flce_fwd_bwd with options (NULL = defaults).  `loss` (host) may be NULL
 * when opts->sync == 0; results then appear in the optional device outputs
 * once `stream` reaches them.  A non-NULL host `loss` forces a synchronous
 * call.
 */
FLCE_API int flce_fwd_bwd_ex(const void* X, const void* W, const int64_t* target, int64_t N, int64_t H,
                    int64_t V, int64_t ignore_index, float* loss, void* dX, float* dW,
                    const flce_opts* opts);

/*
 * Loss only (pass 1 and the row combine; no gradients, no G chunk).  Same
 * arguments and options as flce_fwd_bwd_ex without dX/dW.  Per-row outputs
 * (lse_out, loss_rows_out) make it an evaluation path.
 */
FLCE_API int flce_fwd(const void* X, const void* W, const int64_t* target, int64_t N, int64_t H,
             int64_t V, int64_t ignore_index, float* loss, const flce_opts* opts);

/*
 * Cross-entropy on logits that are already materialised in device memory
 * (the overview's LigerCrossEntropyLoss, "Kernels Básicos"; in-place
 * gradient as in "Operações In-Place"): the same loss and reductions as
 * above with S given directly.
 *   logits [N, V] of element type opts->dtype (bf16 or fp32), row-major
 *   target [N] int64;   loss: host float*, or NULL when opts->sync == 0
 *   dlogits [N, V], same type: dS = valid (softmax - onehot) * grad_scale / n;
 *   it may be the logits buffer itself (the gradient overwrites the logits,
 *   each element after it has been read); NULL computes the loss only.
 * A -inf logit (a masked entry) adds nothing to lse and gets a zero
 * gradient; a row needs one finite logit.  grad_scale may be of any sign;
 * rows whose target is ignore_index get a zero gradient.
 * Optional outputs and error reporting as for flce_fwd_bwd_ex (lse_out,
 * loss_rows_out, loss_dev, n_valid_dev, status_dev, trace).  The scratch
 * space is 12 N bytes plus a few KB.  Memory traffic: one read of the logits
 * from HBM and, with a gradient, one write (the second read of each row
 * comes from shared memory for its last 96 KB, else from L2).
 */
FLCE_API int flce_ce_fwd_bwd(const void* logits, const int64_t* target, int64_t N, int64_t V,
                             int64_t ignore_index, float* loss, void* dlogits,
                             const flce_opts* opts);

/*
 * End-to-end variant on HOST buffers: copies X, W and target to the device,
 * runs the path, and copies loss, dX and dW back.  The W upload goes in
 * pieces on a second stream with pass 1 following piece by piece, and each
 * vocabulary chunk's dW rows are copied back as soon as they are final, while
 * later chunks compute.  Device buffers come from the library's memory pool
 * (stream-ordered).  Pinned host memory gives asynchronous, overlapping
 * copies; pageable memory works but serialises them.  Always synchronous.
 */
FLCE_API int flce_fwd_bwd_host(const void* X_host, const void* W_host, const int64_t* target_host,
                      int64_t N, int64_t H, int64_t V, int64_t ignore_index, float* loss,
                      void* dX_host, float* dW_host, const flce_opts* opts);

/*
 * Scratch bytes a call needs.  with_grads = 0 for flce_fwd, 1 for the
 * gradient entry points.  The plan depends on N, H, V, dtype, vocab_chunk
 * and workspace_budget from `opts` (NULL = defaults).
 */
FLCE_API size_t flce_workspace_bytes(int64_t N, int64_t H, int64_t V, int with_grads,
                            const flce_opts* opts);

/* Static text for a status code. */
FLCE_API const char* flce_status_str(int status);

/* Text of the last error on the calling thread (empty if none). */
FLCE_API const char* flce_last_error(void);

/* FLCE_VERSION of the loaded library. */
FLCE_API int flce_version(void);

/* sizeof(flce_opts) as compiled into the library (lets bindings check their
 * mirror of the struct). */
FLCE_API size_t flce_opts_sizeof(void);

/*
 * Self-test of the kernels' bounded waits (the failure-detection path of
 * every kernel in this library): one block waits on an mbarrier that nothing
 * will arrive on.  The wait must give up after limit_ns nanoseconds (at most
 * 2e9), record the expiry in the status word and let the kernel end
 * normally; the call then returns FLCE_ERR_TIMEOUT, the context stays
 * usable, and later calls work.  Returns FLCE_OK only if the wait did not
 * expire (a fault in the mechanism).  Synchronous; allocates a few bytes.
 */
FLCE_API int flce_selftest_wait_expiry(int64_t limit_ns);

/*
 * Scale and convert a gradient on the device, in one pass over memory:
 *   dst[i] = (dst type)(src[i] * *scale_dev)   (bf16: round to nearest even)
 * This is the step of `loss.backward()` after the overview's
 * loss = loss_fn(weight, input, target) ("Método de API de Baixo Nível"): the
 * gradients were computed in the forward call (dW fp32, dX in the input
 * type), and the backward multiplies them by the incoming grad_output and
 * casts dW to the weight's type.
 *   src [n] of type src_dtype and dst [n] of type dst_dtype (FLCE_BF16 or
 *   FLCE_FP32), device memory; dst may be src itself when the two types are
 *   equal (in place); any other overlap is rejected.
 *   scale_dev: device float (e.g. grad_output), or NULL for 1.
 *   stream: cudaStream_t to launch on (NULL = legacy default stream).
 * Asynchronous.  FLCE_ERR_ARG on n < 0, an unknown type, a null buffer with
 * n > 0, or a forbidden overlap.
 */
FLCE_API int flce_scale_convert(const void* src, int32_t src_dtype, void* dst,
                                int32_t dst_dtype, int64_t n, const float* scale_dev,
                                void* stream);

/*
 * Loss-only pass (the work of flce_fwd) that allocates no device memory.
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc at the point where the loss is needed: a host
 * application that plans all device memory up front in its own arena, a
 * plugin whose execute step may not allocate, or a latency-bound loop where
 * an allocation could synchronise the device or fail under fragmentation.
 *
 * Its scratch space is a static device array inside libflce of
 * 32 MiB (33554432 bytes); every device the library runs on holds it until
 * the process exits.  A problem whose loss-only plan needs more (about
 * 4 * N * ceil(V / 256) + 8 * N bytes plus a few KB; flce_workspace_bytes()
 * with with_grads = 0 gives the exact figure) is rejected with
 * FLCE_ERR_WORKSPACE before anything is launched.
 *
 *   X [N, H], W [V, H] of element type `dtype` (FLCE_BF16 or FLCE_FP32),
 *   target [N] int64: device inputs, read only.
 *   loss_dev (required), lse_out [N], n_valid_dev, status_dev: device outputs
 *   as in flce_opts (NULL skips the optional ones); status_dev receives the
 *   kernels' flce_status (bad targets, expired waits).
 *   stream: cudaStream_t to launch on (NULL = legacy default stream).
 * The call is asynchronous: results are valid once `stream` reaches them.
 *
 * The first call on a device looks up the device address of the static
 * array with cudaGetSymbolAddress (once per device, with that device
 * current); make that first call before any stream capture.  All calls share
 * the one array and each leaves its contents behind: calls that may overlap
 * on the GPU (different streams or host threads without ordering between
 * them) race on it and must be serialised by the caller.
 */
FLCE_API int flce_fwd_noalloc(const void* X, const void* W, const int64_t* target, int64_t N,
                              int64_t H, int64_t V, int64_t ignore_index, int32_t dtype,
                              float* loss_dev, float* lse_out, int64_t* n_valid_dev,
                              int32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
