/*
 * sdpa_oracle.c -- plain fp64 CPU oracle for scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA kernels.
 *
 * What it computes (one query row at a time, nothing larger than one row of
 * scores is ever held):
 *
 *   for every batch b, query head h, query row i:
 *     g    = floor(h / G),   G = Hq / Hkv                     (grouped-query heads)
 *     p_i  = Lk - Lq + i                                      (bottom-right position)
 *     V_i  = { j in [0, Lk) : (!causal or j <= p_i) and (W == 0 or p_i - j < W) }
 *     s_j  = scale * sum_d q[b,h,i,d] * k[b,g,j,d]            (exact fp16/bf16 -> double)
 *            [+ bias[b,h,i,j] when an additive bias (mask array) is given]
 *     P_j  = exp(s_j - max_{V_i} s) / sum_{V_i} exp(s - max s)     for j in V_i, else 0
 *     o[b,h,i,:] = sum_j P_j * v[b,g,j,:]
 *
 * Sources (web pages, by title and section):
 *  - "fix: add head_dim=256 to fused SDPA full attention kernel" (MLX PR #3293),
 *    section "Benchmark: fused vs unfused SDPA for head_dim=256": the unfused
 *    path is "matmul + softmax + matmul"; this oracle is that definition written
 *    row by row.  Its validation test script fixes scale = 1/sqrt(D) and the
 *    (B, H, L, D) array layout.
 *  - "Fused SDPA full-attention for head_dim=192/256" (MLX PR #3660), section
 *    "Microbenchmarks": grouped-query attention with n_q=16, n_kv=8 query/KV
 *    heads; qL < kL workloads.
 *  - "fix: gemma-4 long-prompt prefill OOMs on CUDA ..." (mlxcel issue #672),
 *    sections "Root cause" and "Suggested fix direction": a causal flag and a
 *    windowed causal mask (the dense [L, L] additive mask the page replaces).
 *  - "fix: Gemma 4 MTP never engages on CUDA (GB10) ..." (mlxcel issue #2160),
 *    sections "Current Behavior" (sliding window 1024) and "Proposed Solution"
 *    (a verify row equals a single-row call over the trimmed key prefix, which
 *    fixes the bottom-right alignment p_i = Lk - Lq + i).
 *
 * Readings taken where the pages are silent: causal rows are aligned
 * bottom-right; a window W keeps the W keys j with p_i - j < W (the query's
 * own key included); W = 0 means no window; a window requires causal; query
 * head h reads KV head floor(h / G).  Masked keys are excluded (weight 0), not
 * given a large negative additive value.  An additive bias is added after the
 * scale (as the dense additive mask of mlxcel issue #672 is); a bias entry of
 * -inf removes a key, and a row left with no key outputs zeros.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* IEEE binary16 -> double, exact (every binary16 value is a double). */
static double f16_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)m, -24); /* subnormal: m * 2^-14 * 2^-10 */
  } else if (e == 31) {
    mag = m ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32; widen exactly. */
static double bf16_value(uint16_t b) {
  uint32_t bits = (uint32_t)b << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double elem(const uint16_t *a, int64_t idx, int dtype) {
  return dtype == ORACLE_BF16 ? bf16_value(a[idx]) : f16_value(a[idx]);
}

/* Does query row i (bottom-right position p) see key j? */
static int visible(int64_t j, int64_t p, int causal, int window) {
  if (causal && j > p) return 0;
  if (window > 0 && p - j >= window) return 0;
  return 1;
}

static int check_args(int B, int Hq, int Hkv, int Lq, int Lk, int Dqk, int Dv,
                      int causal, int window, int dtype) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || Dqk <= 0 || Dv <= 0) return -1;
  if (Hq % Hkv != 0) return -1;
  if (window < 0) return -1;
  if (window > 0 && !causal) return -1;
  if (causal && Lq > Lk) return -1; /* a causal row would see no key */
  if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
  return 0;
}

/* Step 1: the scaled scores s_j of row (b, h, i).  With only_visible set, keys
 * outside the row's visible set are skipped (their s_j is left untouched). */
static void row_scores(const uint16_t *q, const uint16_t *k, int dtype, int Hq, int Hkv,
                       int Lq, int Lk, int Dqk, double scale, int b, int h, int i,
                       int only_visible, int causal, int window, double *qrow,
                       double *s, const uint16_t *brow) {
  int G = Hq / Hkv;
  int g = h / G;
  const int64_t qoff = (((int64_t)b * Hq + h) * Lq + i) * Dqk;
  const int64_t kbase = ((int64_t)b * Hkv + g) * (int64_t)Lk * Dqk;
  const int64_t p = (int64_t)Lk - Lq + i;
  for (int d = 0; d < Dqk; ++d) qrow[d] = elem(q, qoff + d, dtype);
  for (int64_t j = 0; j < Lk; ++j) {
    if (only_visible && !visible(j, p, causal, window)) continue;
    double acc = 0.0;
    for (int d = 0; d < Dqk; ++d) acc += qrow[d] * elem(k, kbase + j * Dqk + d, dtype);
    s[j] = scale * acc;
    if (brow) s[j] += elem(brow, j, dtype); /* additive bias (mask array) entry */
  }
}

/* Step 2: softmax over the visible set; P_j = 0 outside it.  Returns -2 if the
 * visible set is empty, 1 (all P_j = 0) if a bias gave every visible key -inf. */
static int row_probs(const double *s, int Lq, int Lk, int i, int causal, int window,
                     double *P) {
  int64_t p = (int64_t)Lk - Lq + i;
  double mx = -INFINITY;
  int any = 0;
  for (int64_t j = 0; j < Lk; ++j)
    if (visible(j, p, causal, window)) {
      any = 1;
      if (s[j] > mx) mx = s[j];
    }
  if (!any) return -2;
  if (mx == -INFINITY) {
    for (int64_t j = 0; j < Lk; ++j) P[j] = 0.0;
    return 1;
  }
  double den = 0.0;
  for (int64_t j = 0; j < Lk; ++j) {
    P[j] = visible(j, p, causal, window) ? exp(s[j] - mx) : 0.0;
    den += P[j];
  }
  for (int64_t j = 0; j < Lk; ++j) P[j] /= den;
  return 0;
}

/* Step 3: o = sum_j P_j v_j. */
static void row_output(const double *P, const uint16_t *v, int dtype, int Hq, int Hkv,
                       int Lk, int Dv, int b, int h, double *o) {
  int G = Hq / Hkv;
  int g = h / G;
  const int64_t vbase = ((int64_t)b * Hkv + g) * (int64_t)Lk * Dv;
  for (int d = 0; d < Dv; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < Lk; ++j) {
    if (P[j] == 0.0) continue;
    for (int d = 0; d < Dv; ++d) o[d] += P[j] * elem(v, vbase + j * Dv + d, dtype);
  }
}

/* Raw scaled scores of one row (step 1 alone), length Lk. */
int oracle_row_scores(const uint16_t *q, const uint16_t *k, int dtype, int B, int Hq,
                      int Hkv, int Lq, int Lk, int Dqk, double scale, int b, int h,
                      int i, double *s_out) {
  if (check_args(B, Hq, Hkv, Lq, Lk, Dqk, Dqk, 0, 0, dtype)) return -1;
  if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Lq) return -1;
  double *qrow = (double *)malloc(sizeof(double) * (size_t)Dqk);
  if (!qrow) return -3;
  row_scores(q, k, dtype, Hq, Hkv, Lq, Lk, Dqk, scale, b, h, i, 0, 0, 0, qrow, s_out, NULL);
  free(qrow);
  return 0;
}

/* Softmax weights of one row (steps 1-2), length Lk, zeros where masked. */
int oracle_row_probs(const uint16_t *q, const uint16_t *k, int dtype, int B, int Hq,
                     int Hkv, int Lq, int Lk, int Dqk, double scale, int causal,
                     int window, int b, int h, int i, double *p_out) {
  if (check_args(B, Hq, Hkv, Lq, Lk, Dqk, Dqk, causal, window, dtype)) return -1;
  if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Lq) return -1;
  double *s = (double *)malloc(sizeof(double) * (size_t)Lk);
  double *qrow = (double *)malloc(sizeof(double) * (size_t)Dqk);
  int rc = -3;
  if (s && qrow) {
    row_scores(q, k, dtype, Hq, Hkv, Lq, Lk, Dqk, scale, b, h, i, 0, causal, window, qrow, s,
               NULL);
    rc = row_probs(s, Lq, Lk, i, causal, window, p_out);
  }
  free(s);
  free(qrow);
  return rc;
}

/*
 * Attention output for a list of rows.  row_ids[r] is the flat row index
 * (b * Hq + h) * Lq + i; when row_ids is NULL, every row in that order
 * (n_rows must then be B * Hq * Lq).  out is n_rows x Dv doubles.
 * nthreads <= 0 lets OpenMP choose.  Returns 0, -1 (bad argument),
 * -2 (a row with no visible key) or -3 (out of memory).
 */
static int sdpa_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const uint16_t *bias, int64_t sb, int64_t sh, int64_t sq, int dtype,
                     int B, int Hq, int Hkv, int Lq, int Lk, int Dqk, int Dv, double scale,
                     int causal, int window, const int64_t *row_ids, int64_t n_rows,
                     double *out, int nthreads) {
  if (check_args(B, Hq, Hkv, Lq, Lk, Dqk, Dv, causal, window, dtype)) return -1;
  const int64_t total = (int64_t)B * Hq * Lq;
  if (n_rows < 0 || (!row_ids && n_rows != total)) return -1;
  if (row_ids)
    for (int64_t r = 0; r < n_rows; ++r)
      if (row_ids[r] < 0 || row_ids[r] >= total) return -1;
  int status = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)Lk);
    double *P = (double *)malloc(sizeof(double) * (size_t)Lk);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)Dqk);
    if (!s || !P || !qrow) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = -3;
    }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < n_rows; ++r) {
      if (!s || !P || !qrow) continue;
      int64_t id = row_ids ? row_ids[r] : r;
      int i = (int)(id % Lq);
      int h = (int)((id / Lq) % Hq);
      int b = (int)(id / ((int64_t)Lq * Hq));
      const uint16_t *brow = bias ? bias + b * sb + h * sh + i * sq : NULL;
      row_scores(q, k, dtype, Hq, Hkv, Lq, Lk, Dqk, scale, b, h, i, 1, causal, window, qrow, s,
                 brow);
      int pr = row_probs(s, Lq, Lk, i, causal, window, P);
      if (pr < 0) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
        status = -2;
        continue;
      }
      row_output(P, v, dtype, Hq, Hkv, Lk, Dv, b, h, out + r * (int64_t)Dv);
    }
    free(s);
    free(P);
    free(qrow);
  }
  return status;
}

int oracle_sdpa(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                int B, int Hq, int Hkv, int Lq, int Lk, int Dqk, int Dv, double scale,
                int causal, int window, const int64_t *row_ids, int64_t n_rows,
                double *out, int nthreads) {
  return sdpa_rows(q, k, v, NULL, 0, 0, 0, dtype, B, Hq, Hkv, Lq, Lk, Dqk, Dv, scale, causal,
                   window, row_ids, n_rows, out, nthreads);
}

/*
 * The same with an additive bias (a mask array): s_j += bias[b*sb + h*sh + i*sq
 * + j], the bias in q's dtype (strides in elements; 0 broadcasts over batch or
 * head).  A bias entry of -inf removes the key; a row whose visible keys all
 * get -inf outputs zeros.
 */
int oracle_sdpa_bias(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const uint16_t *bias, int64_t sb, int64_t sh, int64_t sq, int dtype, int B,
                     int Hq, int Hkv, int Lq, int Lk, int Dqk, int Dv, double scale, int causal,
                     int window, const int64_t *row_ids, int64_t n_rows, double *out,
                     int nthreads) {
  if (!bias || sb < 0 || sh < 0 || sq < 0) return -1;
  return sdpa_rows(q, k, v, bias, sb, sh, sq, dtype, B, Hq, Hkv, Lq, Lk, Dqk, Dv, scale, causal,
                   window, row_ids, n_rows, out, nthreads);
}

/* The thread count OpenMP would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
