/*
 * flce_oracle.c -- plain, slow, double-precision CPU oracle for the fused
 * linear cross-entropy loss and its gradients.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this library.  It shares no
 * code with the CUDA path (no headers, helpers, tables or constants).
 *
 * What it computes (the plain definition; the pages state the loss as
 * loss_fn(weight, input, target) in the Liger-Kernel project overview,
 * "Método de API de Baixo Nível", and say the kernels compute it exactly,
 * "Cálculo Preciso" under "Implementação Técnica"):
 *
 *   S      = X W^T                      X [N,H], W [V,H], S [N,V]
 *   lse_i  = log sum_j exp(S_ij)
 *   valid_i= (t_i != ignore_index),      n_valid = sum_i valid_i
 *   loss   = (1/n_valid) sum_{valid i} (lse_i - S_{i,t_i})      (natural log)
 *   G_ij   = valid_i (exp(S_ij - lse_i) - [j == t_i]) / n_valid
 *   dX     = G W,   dW = G^T X
 *
 * Readings taken where the pages are silent: mean over valid rows; when
 * n_valid == 0 the loss and both gradients are 0; a target outside [0, V)
 * that is not the ignore index is an error (return code 2).  A call that is
 * one data-parallel shard of a larger batch (the overview's FSDP / DeepSpeed
 * compatibility, "Alta Compatibilidade") may give the whole batch's valid
 * count as norm_count > 0: the mean and G are then divided by it instead of
 * by this call's own count, so the shards' losses, dW and dX rows add up to
 * the whole batch's.
 *
 * Arithmetic: every product and sum in double, in the order written below
 * (sums over H and V run from index 0 upward).  The max-shift inside lse is
 * the usual stabiliser log sum exp(S) = m + log sum exp(S - m) with
 * m = max_j S_ij; it changes no value beyond rounding.
 *
 * Layout: row-major, contiguous.  Input element types: 0 = float64,
 * 1 = float32, 2 = bfloat16 given as its 16 raw bits (widened exactly).
 * Parallelism: OpenMP over independent rows / vocabulary entries only; each
 * output element has one writer, so results do not depend on thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };


static double bf16_to_double(uint16_t v) {
  uint32_t bits = (uint32_t)v << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double elem(const void *p, int type, int64_t i) {
  if (type == ORC_F64) return ((const double *)p)[i];
  if (type == ORC_F32) return (double)((const float *)p)[i];
  /* bfloat16: the upper 16 bits of an IEEE float32 */
  return bf16_to_double(((const uint16_t *)p)[i]);
}

/* S_ij = sum_h X[i,h] * W[j,h]  (one loop per element type; same order) */
static double logit(const void *X, const void *W, int type, int64_t H,
                    int64_t i, int64_t j) {
  double s = 0.0;
  if (type == ORC_F64) {
    const double *x = (const double *)X + i * H, *w = (const double *)W + j * H;
    for (int64_t h = 0; h < H; ++h) s += x[h] * w[h];
  } else if (type == ORC_F32) {
    const float *x = (const float *)X + i * H, *w = (const float *)W + j * H;
    for (int64_t h = 0; h < H; ++h) s += (double)x[h] * (double)w[h];
  } else {
    const uint16_t *x = (const uint16_t *)X + i * H, *w = (const uint16_t *)W + j * H;
    for (int64_t h = 0; h < H; ++h) s += bf16_to_double(x[h]) * bf16_to_double(w[h]);
  }
  return s;
}

/* Row i of S into srow[V]. */
static void logit_row(const void *X, const void *W, int type, int64_t H,
                      int64_t V, int64_t i, double *srow) {
  for (int64_t j = 0; j < V; ++j) srow[j] = logit(X, W, type, H, i, j);
}

/* log sum_j exp(srow[j]) */
static double logsumexp(const double *srow, int64_t V) {
  double m = -INFINITY;
  for (int64_t j = 0; j < V; ++j)
    if (srow[j] > m) m = srow[j];
  double s = 0.0;
  for (int64_t j = 0; j < V; ++j) s += exp(srow[j] - m);
  return m + log(s);
}

int64_t oracle_count_valid(const int64_t *t, int64_t N, int64_t ignore_index) {
  int64_t n = 0;
  for (int64_t i = 0; i < N; ++i) n += (t[i] != ignore_index);
  return n;
}

/* 0 = ok, 1 = bad arguments, 2 = a target outside [0, V) that is not ignored */
static int check_targets(const int64_t *t, int64_t N, int64_t V,
                         int64_t ignore_index) {
  for (int64_t i = 0; i < N; ++i)
    if (t[i] != ignore_index && (t[i] < 0 || t[i] >= V)) return 2;
  return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Full problem.  Outputs: *loss, *n_valid, lse[N] (may be NULL),
 * loss_rows[N] per-row lse_i - S_{i,t_i} (0 for ignored rows; may be NULL),
 * dX[N*H] and dW[V*H] (either may be NULL to skip it).  norm_count <= 0
 * divides by this call's valid count n_valid; norm_count > 0 divides by it
 * instead (a shard of a larger batch).
 */
int oracle_flce(const void *X, const void *W, int type, const int64_t *t,
                int64_t N, int64_t H, int64_t V, int64_t ignore_index,
                int64_t norm_count, double *loss, int64_t *n_valid, double *lse,
                double *loss_rows, double *dX, double *dW) {
  if (N < 0 || H <= 0 || V <= 0 || !loss || !n_valid) return 1;
  if (N > 0 && (!X || !W || !t)) return 1;
  int rc = check_targets(t, N, V, ignore_index);
  if (rc) return rc;
  const int64_t nv = oracle_count_valid(t, N, ignore_index);
  *n_valid = nv;
  const double den = norm_count > 0 ? (double)norm_count : (double)nv;

  double *lse_all = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
  double *lrow = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
  if (!lse_all || !lrow) { free(lse_all); free(lrow); return 1; }

  /* Phase A: per row, lse_i and the row loss lse_i - S_{i,t_i}. */
#pragma omp parallel
  {
    double *srow = (double *)malloc((size_t)V * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < N; ++i) {
      logit_row(X, W, type, H, V, i, srow);
      lse_all[i] = logsumexp(srow, V);
      lrow[i] = (t[i] != ignore_index) ? lse_all[i] - srow[t[i]] : 0.0;
    }
    free(srow);
  }

  /* loss: ordered sum over rows, then the mean over valid rows */
  double acc = 0.0;
  for (int64_t i = 0; i < N; ++i) acc += lrow[i];
  *loss = nv > 0 ? acc / den : 0.0;
  if (lse) memcpy(lse, lse_all, (size_t)N * sizeof(double));
  if (loss_rows) memcpy(loss_rows, lrow, (size_t)N * sizeof(double));

  /* Phase B: dW_j = sum_i G_ij x_i, one vocabulary row per task. */
  if (dW) {
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t j = 0; j < V; ++j) {
      double *dwj = dW + j * H;
      for (int64_t h = 0; h < H; ++h) dwj[h] = 0.0;
      if (nv == 0) continue;
      for (int64_t i = 0; i < N; ++i) {
        if (t[i] == ignore_index) continue;
        double g = exp(logit(X, W, type, H, i, j) - lse_all[i]) -
                   (t[i] == j ? 1.0 : 0.0);
        g /= den;
        for (int64_t h = 0; h < H; ++h) dwj[h] += g * elem(X, type, i * H + h);
      }
    }
  }

  /* Phase C: dX_i = sum_j G_ij w_j, one token row per task. */
  if (dX) {
#pragma omp parallel
    {
      double *srow = (double *)malloc((size_t)V * sizeof(double));
#pragma omp for schedule(dynamic, 1)
      for (int64_t i = 0; i < N; ++i) {
        double *dxi = dX + i * H;
        for (int64_t h = 0; h < H; ++h) dxi[h] = 0.0;
        if (t[i] == ignore_index || nv == 0) continue;
        logit_row(X, W, type, H, V, i, srow);
        for (int64_t j = 0; j < V; ++j) {
          double g = exp(srow[j] - lse_all[i]) - (t[i] == j ? 1.0 : 0.0);
          g /= den;
          for (int64_t h = 0; h < H; ++h) dxi[h] += g * elem(W, type, j * H + h);
        }
      }
      free(srow);
    }
  }
  free(lse_all);
  free(lrow);
  return 0;
}

/*
 * Selected token rows of the full problem (the normaliser n_valid is still
 * counted over all N targets).  For each rows[r]: lse, the row loss and, if
 * dX_rows is not NULL, dX row (H values).  Cost: two passes over W per row.
 */
int oracle_flce_rows(const void *X, const void *W, int type, const int64_t *t,
                     int64_t N, int64_t H, int64_t V, int64_t ignore_index,
                     const int64_t *rows, int64_t n_rows, double *lse_rows,
                     double *loss_rows, double *dX_rows, int64_t *n_valid) {
  if (N <= 0 || H <= 0 || V <= 0 || !X || !W || !t || !rows) return 1;
  int rc = check_targets(t, N, V, ignore_index);
  if (rc) return rc;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return 1;
  const int64_t nv = oracle_count_valid(t, N, ignore_index);
  if (n_valid) *n_valid = nv;
#pragma omp parallel
  {
    double *srow = (double *)malloc((size_t)V * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
      const int64_t i = rows[r];
      logit_row(X, W, type, H, V, i, srow);
      const double l = logsumexp(srow, V);
      const int valid = t[i] != ignore_index;
      if (lse_rows) lse_rows[r] = l;
      if (loss_rows) loss_rows[r] = valid ? l - srow[t[i]] : 0.0;
      if (dX_rows) {
        double *dxi = dX_rows + r * H;
        for (int64_t h = 0; h < H; ++h) dxi[h] = 0.0;
        if (valid && nv > 0) {
          for (int64_t j = 0; j < V; ++j) {
            double g = (exp(srow[j] - l) - (t[i] == j ? 1.0 : 0.0)) / (double)nv;
            for (int64_t h = 0; h < H; ++h) dxi[h] += g * elem(W, type, j * H + h);
          }
        }
      }
    }
    free(srow);
  }
  return 0;
}

/*
 * Selected vocabulary rows of dW for the full problem: dW_j = sum_i G_ij x_i
 * for j in vocab[].  Needs lse for every token row first (cost N*V*H).
 */
int oracle_flce_dw_rows(const void *X, const void *W, int type, const int64_t *t,
                        int64_t N, int64_t H, int64_t V, int64_t ignore_index,
                        const int64_t *vocab, int64_t n_vocab, double *dW_rows) {
  if (N < 0 || H <= 0 || V <= 0 || !vocab || !dW_rows) return 1;
  int rc = check_targets(t, N, V, ignore_index);
  if (rc) return rc;
  for (int64_t r = 0; r < n_vocab; ++r)
    if (vocab[r] < 0 || vocab[r] >= V) return 1;
  const int64_t nv = oracle_count_valid(t, N, ignore_index);
  double *lse_all = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
  if (!lse_all) return 1;
#pragma omp parallel
  {
    double *srow = (double *)malloc((size_t)V * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < N; ++i) {
      logit_row(X, W, type, H, V, i, srow);
      lse_all[i] = logsumexp(srow, V);
    }
    free(srow);
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_vocab; ++r) {
    const int64_t j = vocab[r];
    double *dwj = dW_rows + r * H;
    for (int64_t h = 0; h < H; ++h) dwj[h] = 0.0;
    if (nv == 0) continue;
    for (int64_t i = 0; i < N; ++i) {
      if (t[i] == ignore_index) continue;
      double g = (exp(logit(X, W, type, H, i, j) - lse_all[i]) -
                  (t[i] == j ? 1.0 : 0.0)) / (double)nv;
      for (int64_t h = 0; h < H; ++h) dwj[h] += g * elem(X, type, i * H + h);
    }
  }
  free(lse_all);
  return 0;
}

/*
 * Cross-entropy on logits that are already materialised (the operator the
 * overview lists as LigerCrossEntropyLoss, "Kernels Básicos"): the same
 * definition as above with S given directly as an [N, V] matrix.
 *   loss = (1/n) sum_{valid i} (lse_i - S_{i,t_i}),
 *   dS_ij = valid_i (exp(S_ij - lse_i) - [j == t_i]) / n
 * Outputs: *loss, *n_valid, lse[N], loss_rows[N] (may be NULL), dS[N*V]
 * (may be NULL).  Element types as for oracle_flce.
 */
int oracle_ce(const void *S, int type, const int64_t *t, int64_t N, int64_t V,
              int64_t ignore_index, double *loss, int64_t *n_valid, double *lse,
              double *loss_rows, double *dS) {
  if (N < 0 || V <= 0 || !loss || !n_valid) return 1;
  if (N > 0 && (!S || !t)) return 1;
  int rc = check_targets(t, N, V, ignore_index);
  if (rc) return rc;
  const int64_t nv = oracle_count_valid(t, N, ignore_index);
  *n_valid = nv;
  double *lrow = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
  if (!lrow) return 1;
#pragma omp parallel
  {
    double *srow = (double *)malloc((size_t)V * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < N; ++i) {
      for (int64_t j = 0; j < V; ++j) srow[j] = elem(S, type, i * V + j);
      const double l = logsumexp(srow, V);
      const int valid = t[i] != ignore_index;
      if (lse) lse[i] = l;
      lrow[i] = valid ? l - srow[t[i]] : 0.0;
      if (dS) {
        for (int64_t j = 0; j < V; ++j) {
          double g = 0.0;
          if (valid && nv > 0)
            g = (exp(srow[j] - l) - (t[i] == j ? 1.0 : 0.0)) / (double)nv;
          dS[i * V + j] = g;
        }
      }
    }
    free(srow);
  }
  double acc = 0.0;
  for (int64_t i = 0; i < N; ++i) acc += lrow[i];
  *loss = nv > 0 ? acc / (double)nv : 0.0;
  if (loss_rows) memcpy(loss_rows, lrow, (size_t)N * sizeof(double));
  free(lrow);
  return 0;
}
