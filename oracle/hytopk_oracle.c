/*
 * hytopk_oracle.c -- CPU oracle for exact per-query top-k selection over
 * DeepSeek-style indexer scores, for the threshold filter that HyTopK runs
 * in front of that selection, and for selection replay.
 *
 * TEST INFRASTRUCTURE ONLY. This is the plain, slow, obviously correct
 * definition that the GPU library is checked against. Only the tests, the
 * package's smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (web pages on HyScale; cited by title and paragraph):
 *   [Summary]   "HyScale: Scaling Long-Context Training for Learned Sparse
 *               Attention" (neuraltrendhub), "What the paper found" and
 *               "Original abstract".
 *   [Explainer] "HyScale sparse-attention training -- Selection without a
 *               score table -- What does it mean?" (learnaivisually): the
 *               score-table paragraph, the HyTopK paragraph, the selection
 *               replay paragraph and the worked GLM-5.1 example.
 *
 * What is computed (readings of the pages are marked READING):
 *   ctx(t) = positions[t] + 1: query t sees keys s <= positions[t]
 *     (each query scores all tokens before it: Summary, What the paper found).
 *   I[t,s] = sum_h w[t,h] * max(0, dot_h),  dot_h = sum_i q[t,h,i] * k[s,i]
 *     READING: the DeepSeek-style indexer score (Summary names DeepSeek-style
 *     token selection; Explainer, score-table paragraph, calls it attention-
 *     score work that is cheaper per token). One shared key head.
 *   Arithmetic is fp32 with sequential summation (dot over i = 0..d-1, then
 *     the weighted sum over h = 0..H-1), one rounding per operation: the
 *     file must be compiled with -ffp-contract=off so no multiply-add is
 *     fused and x86 and Arm give the same bits.
 *   Inputs: bf16 (bit shift to fp32) or OCP FP8 E4M3 ("fn": bias 7, no
 *     infinities, S.1111.111 is NaN, max 448) times an fp32 scale per
 *     128-element row: q_scale[t,h], k_scale[s]. The scale is applied to the
 *     element before the dot. dtype 2 is e4m3 q (with q_scale) and bf16 k
 *     (without a scale).
 *   -0.0 scores are canonicalised to +0.0.
 *   Exact top-k (Explainer, HyTopK paragraph): order all (I, s), s < ctx, by
 *     I descending, then s ascending (READING: the lower position wins a tie
 *     at the k-th score; the output is sorted in that order), emit the first
 *     min(k, ctx) positions and pad with -1 (scores pad with -inf).
 *   Threshold filter (Explainer, HyTopK paragraph and worked example):
 *     M = min(ctx, max(4096, floor(ctx/128)), 8192) evenly spaced samples
 *     p_j = floor(j*ctx/M) (READING: offset 0, floor), threshold T = the r-th
 *     largest sample score counting ties, r = min(M, ceil(3*k*M/ctx)); keys
 *     with I >= T are candidates; a query with ctx > k fails when it has fewer
 *     than k candidates or more than the buffer capacity C.
 *   Replay (Explainer, selection replay paragraph): the same score at stored
 *     indices; index -1 gives -inf, any other index outside [0, L) gives NaN
 *     and is counted as bad.
 *   Backward at the selected entries (Explainer, key-observation paragraph:
 *     the indexer's own loss reads only the scores at the selected entries;
 *     selection-replay paragraph: those entries are rescored during
 *     recomputation). Given G[t,j] = dLoss/dI[t, idx[t,j]] (READING: the loss
 *     itself is not on the pages, so its gradient is an input), with the
 *     dequantised inputs qd = q*q_scale and kd = k*k_scale, x = qd[t,h].kd[s]:
 *       dw[t,h]   = sum_j G[t,j] * max(0, x[t,h,idx[t,j]])
 *       dq[t,h,:] = sum_j G[t,j] * w[t,h] * [x > 0] * kd[idx[t,j],:]
 *       dk[s,:]  += sum_{(t,j): idx[t,j] = s} G[t,j] * sum_h w[t,h] * [x > 0] * qd[t,h,:]
 *     READING: the derivative of max(0, x) at x = 0 is taken as 0. This part
 *     is computed in fp64 (the pages fix no precision for it).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BF16 0
#define ORACLE_E4M3 1
#define ORACLE_E4M3_BF16 2 /* q e4m3 with q_scale, k bf16 without a scale */

static int q_dtype(int dtype) { return dtype == ORACLE_BF16 ? ORACLE_BF16 : ORACLE_E4M3; }
static int k_dtype(int dtype) { return dtype == ORACLE_E4M3 ? ORACLE_E4M3 : ORACLE_BF16; }
static int valid_dtype(int dtype) { return dtype >= ORACLE_BF16 && dtype <= ORACLE_E4M3_BF16; }

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_POSITION 2
#define ORACLE_NO_MEMORY 3

/* ---- element decoding, from the format definitions ---------------------- */

/* bf16 is the top half of an IEEE binary32. */
float oracle_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* OCP FP8 E4M3 (fn): sign, 4 exponent bits with bias 7, 3 mantissa bits.
 * Exponent field 0 is subnormal (m/8 * 2^-6); 1111 with mantissa 111 is NaN;
 * there is no infinity, so 1111 with mantissa 000..110 are normal numbers. */
float oracle_e4m3_value(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return (float)NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* (m/8) * 2^(1-7) */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return (float)(sign ? -v : v);
}

void oracle_e4m3_table(float* out256) {
  for (int c = 0; c < 256; ++c) out256[c] = oracle_e4m3_value((uint8_t)c);
}

/* ---- threshold parameters (Explainer, HyTopK paragraph, worked example) --- */

int64_t oracle_sample_count(int64_t ctx) {
  int64_t m = ctx / 128;
  if (m < 4096) m = 4096;
  if (m > 8192) m = 8192;
  if (m > ctx) m = ctx;
  return m;
}

int64_t oracle_threshold_rank(int64_t ctx, int64_t k_top) {
  int64_t m = oracle_sample_count(ctx);
  if (ctx <= 0) return 0;
  int64_t r = (3 * k_top * m + ctx - 1) / ctx; /* ceil(3kM/ctx) */
  return r < m ? r : m;
}

int64_t oracle_sample_position(int64_t ctx, int64_t m, int64_t j) {
  return (j * ctx) / m; /* floor, non-negative operands */
}

void oracle_sample_positions(int64_t ctx, int64_t* out) {
  int64_t m = oracle_sample_count(ctx);
  for (int64_t j = 0; j < m; ++j) out[j] = oracle_sample_position(ctx, m, j);
}

/* ---- the problem -------------------------------------------------------- */

typedef struct {
  const void* q;        /* [n,H,d] bf16 bits or e4m3 codes */
  const float* q_scale; /* [n,H] (e4m3) or NULL */
  const void* k;        /* [L,d] */
  const float* k_scale; /* [L] (e4m3) or NULL */
  const float* w;       /* [n,H] */
  const int32_t* positions;
  int64_t n, L;
  int H, d, dtype;
  float* kf; /* decoded keys [L][d] with the scale applied */
} problem;

static float element(const void* base, int dtype, size_t i) {
  if (dtype == ORACLE_BF16) return oracle_bf16_value(((const uint16_t*)base)[i]);
  return oracle_e4m3_value(((const uint8_t*)base)[i]);
}

static int setup(problem* p) {
  size_t L = (size_t)p->L, d = (size_t)p->d;
  if (p->L <= 0 || p->H <= 0 || p->d <= 0 || p->n < 0) return ORACLE_BAD_ARG;
  if (!valid_dtype(p->dtype)) return ORACLE_BAD_ARG;
  if (q_dtype(p->dtype) == ORACLE_E4M3 && !p->q_scale) return ORACLE_BAD_ARG;
  if (k_dtype(p->dtype) == ORACLE_E4M3 && !p->k_scale) return ORACLE_BAD_ARG;
  p->kf = (float*)malloc(L * d * sizeof(float));
  if (!p->kf) return ORACLE_NO_MEMORY;
#pragma omp parallel for schedule(static)
  for (int64_t s = 0; s < p->L; ++s) {
    const int kd = k_dtype(p->dtype);
    float scale = kd == ORACLE_E4M3 ? p->k_scale[s] : 1.0f;
    for (size_t i = 0; i < d; ++i) {
      float v = element(p->k, kd, (size_t)s * d + i);
      p->kf[(size_t)s * d + i] = kd == ORACLE_E4M3 ? v * scale : v;
    }
  }
  return ORACLE_OK;
}

/* Query t's operand, transposed to [d][H] so that the inner loop over heads
 * runs over independent accumulators (each dot still sums i = 0..d-1 in
 * order). */
static void query_operand(const problem* p, int64_t t, float* qT) {
  for (int h = 0; h < p->H; ++h) {
    const int qd = q_dtype(p->dtype);
    float scale = qd == ORACLE_E4M3 ? p->q_scale[t * p->H + h] : 1.0f;
    for (int i = 0; i < p->d; ++i) {
      size_t at = ((size_t)t * p->H + h) * p->d + i;
      float v = element(p->q, qd, at);
      qT[(size_t)i * p->H + h] = qd == ORACLE_E4M3 ? v * scale : v;
    }
  }
}

/* I[t,s] for one key; dot is scratch of H floats. */
static float score_one(const problem* p, const float* qT, const float* wt, int64_t s,
                       float* dot) {
  const int H = p->H, d = p->d;
  const float* kr = p->kf + (size_t)s * d;
  for (int h = 0; h < H; ++h) dot[h] = 0.0f;
  for (int i = 0; i < d; ++i) {
    const float ki = kr[i];
    const float* qi = qT + (size_t)i * H;
    for (int h = 0; h < H; ++h) dot[h] += qi[h] * ki;
  }
  float acc = 0.0f;
  for (int h = 0; h < H; ++h) {
    float relu = dot[h] > 0.0f ? dot[h] : 0.0f;
    acc += wt[h] * relu;
  }
  if (acc == 0.0f) acc = 0.0f; /* -0.0 -> +0.0 */
  return acc;
}

typedef struct {
  float score;
  int32_t pos;
} entry;

/* score descending, then position ascending */
static int entry_order(const void* a, const void* b) {
  const entry* x = (const entry*)a;
  const entry* y = (const entry*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->pos > y->pos) - (x->pos < y->pos);
}

static int descending_float(const void* a, const void* b) {
  float x = *(const float*)a, y = *(const float*)b;
  return (x < y) - (x > y);
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

static int check_positions(const problem* p, const int32_t* rows, int64_t n_rows) {
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t t = rows ? rows[r] : r;
    if (t < 0 || t >= p->n) return ORACLE_BAD_ARG;
    if (p->positions[t] < 0 || p->positions[t] >= p->L) return ORACLE_BAD_POSITION;
  }
  return ORACLE_OK;
}

/* Every score of query t over its causal prefix: out[s], s < ctx(t). */
int oracle_row_scores(const void* q, const float* q_scale, const void* k, const float* k_scale,
                      const float* w, const int32_t* positions, int64_t n, int64_t L, int H,
                      int d, int dtype, int64_t t, float* out, int nthreads) {
  problem p = {q, q_scale, k, k_scale, w, positions, n, L, H, d, dtype, NULL};
  int32_t row = (int32_t)t;
  int st = setup(&p);
  if (st) return st;
  st = check_positions(&p, &row, 1);
  if (st) {
    free(p.kf);
    return st;
  }
  set_threads(nthreads);
  int64_t ctx = (int64_t)positions[t] + 1;
  float* qT = (float*)malloc((size_t)H * d * sizeof(float));
  query_operand(&p, t, qT);
#pragma omp parallel
  {
    float* dot = (float*)malloc((size_t)H * sizeof(float));
#pragma omp for schedule(static)
    for (int64_t s = 0; s < ctx; ++s) out[s] = score_one(&p, qT, w + (size_t)t * H, s, dot);
    free(dot);
  }
  free(qT);
  free(p.kf);
  return ORACLE_OK;
}

/* Exact top-k of each listed query (rows == NULL: all n queries, in order).
 * idx_out/scores_out: [n_rows, k_top]. */
int oracle_select(const void* q, const float* q_scale, const void* k, const float* k_scale,
                  const float* w, const int32_t* positions, const int32_t* rows, int64_t n_rows,
                  int64_t n, int64_t L, int H, int d, int dtype, int64_t k_top,
                  int32_t* idx_out, float* scores_out, int nthreads) {
  problem p = {q, q_scale, k, k_scale, w, positions, n, L, H, d, dtype, NULL};
  if (k_top <= 0 || n_rows < 0) return ORACLE_BAD_ARG;
  int st = setup(&p);
  if (st) return st;
  st = check_positions(&p, rows, n_rows);
  if (st) {
    free(p.kf);
    return st;
  }
  set_threads(nthreads);
#pragma omp parallel
  {
    float* qT = (float*)malloc((size_t)H * d * sizeof(float));
    float* dot = (float*)malloc((size_t)H * sizeof(float));
    entry* all = (entry*)malloc((size_t)L * sizeof(entry));
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
      int64_t t = rows ? rows[r] : r;
      int64_t ctx = (int64_t)positions[t] + 1;
      query_operand(&p, t, qT);
      for (int64_t s = 0; s < ctx; ++s) {
        all[s].score = score_one(&p, qT, w + (size_t)t * H, s, dot);
        all[s].pos = (int32_t)s;
      }
      qsort(all, (size_t)ctx, sizeof(entry), entry_order);
      for (int64_t j = 0; j < k_top; ++j) {
        int keep = j < ctx;
        idx_out[r * k_top + j] = keep ? all[j].pos : -1;
        if (scores_out) scores_out[r * k_top + j] = keep ? all[j].score : -INFINITY;
      }
    }
    free(all);
    free(dot);
    free(qT);
  }
  free(p.kf);
  return ORACLE_OK;
}

/* Selection replay: out[t,j] = I[t, idx[t,j]]. Returns the number of
 * out-of-range indices through *bad (those entries are NaN). */
int oracle_replay(const void* q, const float* q_scale, const void* k, const float* k_scale,
                  const float* w, const int32_t* idx, int64_t n, int64_t L, int H, int d,
                  int dtype, int64_t k_top, float* out, int64_t* bad, int nthreads) {
  problem p = {q, q_scale, k, k_scale, w, NULL, n, L, H, d, dtype, NULL};
  int64_t nbad = 0;
  if (k_top <= 0) return ORACLE_BAD_ARG;
  int st = setup(&p);
  if (st) return st;
  set_threads(nthreads);
#pragma omp parallel reduction(+ : nbad)
  {
    float* qT = (float*)malloc((size_t)H * d * sizeof(float));
    float* dot = (float*)malloc((size_t)H * sizeof(float));
#pragma omp for schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
      query_operand(&p, t, qT);
      for (int64_t j = 0; j < k_top; ++j) {
        int32_t s = idx[t * k_top + j];
        float v;
        if (s == -1)
          v = -INFINITY;
        else if (s < 0 || s >= L) {
          v = NAN;
          ++nbad;
        } else
          v = score_one(&p, qT, w + (size_t)t * H, s, dot);
        out[t * k_top + j] = v;
      }
    }
    free(dot);
    free(qT);
  }
  free(p.kf);
  if (bad) *bad = nbad;
  return ORACLE_OK;
}

/* The threshold filter, simulated from its definition: per listed query the
 * sample count M, rank r, threshold T, candidate count and failed flag.
 * Queries with ctx <= k select everything: M = r = 0, T = -inf, cnt = ctx,
 * never failed. */
int oracle_filter_sim(const void* q, const float* q_scale, const void* k, const float* k_scale,
                      const float* w, const int32_t* positions, const int32_t* rows,
                      int64_t n_rows, int64_t n, int64_t L, int H, int d, int dtype,
                      int64_t k_top, int64_t capacity, float* T_out, int64_t* cnt_out,
                      int64_t* M_out, int64_t* r_out, uint8_t* failed_out, int nthreads) {
  problem p = {q, q_scale, k, k_scale, w, positions, n, L, H, d, dtype, NULL};
  if (k_top <= 0 || capacity < k_top || n_rows < 0) return ORACLE_BAD_ARG;
  int st = setup(&p);
  if (st) return st;
  st = check_positions(&p, rows, n_rows);
  if (st) {
    free(p.kf);
    return st;
  }
  set_threads(nthreads);
#pragma omp parallel
  {
    float* qT = (float*)malloc((size_t)H * d * sizeof(float));
    float* dot = (float*)malloc((size_t)H * sizeof(float));
    float* row = (float*)malloc((size_t)L * sizeof(float));
    float* samp = (float*)malloc(8192 * sizeof(float));
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
      int64_t t = rows ? rows[r] : r;
      int64_t ctx = (int64_t)positions[t] + 1;
      query_operand(&p, t, qT);
      for (int64_t s = 0; s < ctx; ++s) row[s] = score_one(&p, qT, w + (size_t)t * H, s, dot);
      if (ctx <= k_top) {
        T_out[r] = -INFINITY;
        cnt_out[r] = ctx;
        M_out[r] = 0;
        r_out[r] = 0;
        failed_out[r] = 0;
        continue;
      }
      int64_t m = oracle_sample_count(ctx);
      int64_t rank = oracle_threshold_rank(ctx, k_top);
      for (int64_t j = 0; j < m; ++j) samp[j] = row[oracle_sample_position(ctx, m, j)];
      qsort(samp, (size_t)m, sizeof(float), descending_float);
      float T = samp[rank - 1];
      int64_t cnt = 0;
      for (int64_t s = 0; s < ctx; ++s) cnt += row[s] >= T;
      T_out[r] = T;
      cnt_out[r] = cnt;
      M_out[r] = m;
      r_out[r] = rank;
      failed_out[r] = (uint8_t)(cnt < k_top || cnt > capacity);
    }
    free(samp);
    free(row);
    free(dot);
    free(qT);
  }
  free(p.kf);
  return ORACLE_OK;
}

/* Backward of sum_{t,j} G[t,j] * I[t, idx[t,j]] (see the header): outputs in
 * fp64, dq [n,H,d] and dw [n,H] written, dk [L,d] accumulated into. For
 * tolerances it also returns, per output element, the sum of the absolute
 * values of its terms (*_abs) and the part of that sum whose head dot x lies
 * within eps * |qd[t,h]| * |kd[s]| of zero (*_amb: terms whose [x > 0]
 * depends on rounding). Any of the *_abs / *_amb arrays may be NULL.
 * Entries with idx = -1 contribute nothing; other indices outside [0, L) are
 * counted in *bad and skipped. */
int oracle_backward(const void* q, const float* q_scale, const void* k, const float* k_scale,
                    const float* w, const int32_t* idx, const float* grad, int64_t n, int64_t L,
                    int H, int d, int dtype, int64_t k_top, double eps, double* dq, double* dk,
                    double* dw, double* dq_abs, double* dk_abs, double* dw_abs, double* dq_amb,
                    double* dk_amb, double* dw_amb, int64_t* bad, int nthreads) {
  if (n < 0 || L <= 0 || H <= 0 || d <= 0 || k_top <= 0) return ORACLE_BAD_ARG;
  if (!valid_dtype(dtype)) return ORACLE_BAD_ARG;
  if (q_dtype(dtype) == ORACLE_E4M3 && !q_scale) return ORACLE_BAD_ARG;
  if (k_dtype(dtype) == ORACLE_E4M3 && !k_scale) return ORACLE_BAD_ARG;
  const size_t Hd = (size_t)H * d;
  /* dequantised keys and their norms, fp64 (the products are exact) */
  double* kd = (double*)malloc((size_t)L * d * sizeof(double));
  double* knorm = (double*)malloc((size_t)L * sizeof(double));
  if (!kd || !knorm) {
    free(kd);
    free(knorm);
    return ORACLE_NO_MEMORY;
  }
  set_threads(nthreads);
#pragma omp parallel for schedule(static)
  for (int64_t s = 0; s < L; ++s) {
    double scale = k_dtype(dtype) == ORACLE_E4M3 ? (double)k_scale[s] : 1.0;
    double nn = 0.0;
    for (int i = 0; i < d; ++i) {
      double v = (double)element(k, k_dtype(dtype), (size_t)s * d + i) * scale;
      kd[(size_t)s * d + i] = v;
      nn += v * v;
    }
    knorm[s] = sqrt(nn);
  }
  int64_t nbad = 0;
  for (int64_t t = 0; t < n; ++t)
    for (int64_t j = 0; j < k_top; ++j) {
      int32_t s = idx[t * k_top + j];
      if (s != -1 && (s < 0 || s >= L)) ++nbad;
    }
  /* dq and dw: one query at a time (independent) */
#pragma omp parallel
  {
    double* qd = (double*)malloc(Hd * sizeof(double));
    double* qnorm = (double*)malloc((size_t)H * sizeof(double));
#pragma omp for schedule(dynamic, 4)
    for (int64_t t = 0; t < n; ++t) {
      for (int h = 0; h < H; ++h) {
        double scale = q_dtype(dtype) == ORACLE_E4M3 ? (double)q_scale[t * H + h] : 1.0;
        double nn = 0.0;
        for (int i = 0; i < d; ++i) {
          double v = (double)element(q, q_dtype(dtype), ((size_t)t * H + h) * d + i) * scale;
          qd[(size_t)h * d + i] = v;
          nn += v * v;
        }
        qnorm[h] = sqrt(nn);
      }
      double* dqt = dq + (size_t)t * Hd;
      for (size_t e = 0; e < Hd; ++e) {
        dqt[e] = 0.0;
        if (dq_abs) dq_abs[(size_t)t * Hd + e] = 0.0;
        if (dq_amb) dq_amb[(size_t)t * Hd + e] = 0.0;
      }
      for (int h = 0; h < H; ++h) {
        dw[t * H + h] = 0.0;
        if (dw_abs) dw_abs[t * H + h] = 0.0;
        if (dw_amb) dw_amb[t * H + h] = 0.0;
      }
      for (int64_t j = 0; j < k_top; ++j) {
        int32_t s = idx[t * k_top + j];
        if (s < 0 || s >= L) continue;
        double g = (double)grad[t * k_top + j];
        const double* ks = kd + (size_t)s * d;
        for (int h = 0; h < H; ++h) {
          double x = 0.0;
          for (int i = 0; i < d; ++i) x += qd[(size_t)h * d + i] * ks[i];
          int amb = fabs(x) <= eps * qnorm[h] * knorm[s];
          double relu = x > 0.0 ? x : 0.0;
          dw[t * H + h] += g * relu;
          if (dw_abs) dw_abs[t * H + h] += fabs(g * relu);
          if (dw_amb && amb) dw_amb[t * H + h] += fabs(g * x);
          double coef = g * (double)w[t * H + h];
          for (int i = 0; i < d; ++i) {
            size_t e = (size_t)h * d + i;
            if (x > 0.0) {
              dqt[e] += coef * ks[i];
              if (dq_abs) dq_abs[(size_t)t * Hd + e] += fabs(coef * ks[i]);
            }
            if (dq_amb && amb) dq_amb[(size_t)t * Hd + e] += fabs(coef * ks[i]);
          }
        }
      }
    }
    free(qnorm);
    free(qd);
  }
  /* dk: every (query, entry) adds into its key's row, in query order */
  double* qd = (double*)malloc(Hd * sizeof(double));
  double* qnorm = (double*)malloc((size_t)H * sizeof(double));
  for (int64_t t = 0; t < n && qd && qnorm; ++t) {
    for (int h = 0; h < H; ++h) {
      double scale = q_dtype(dtype) == ORACLE_E4M3 ? (double)q_scale[t * H + h] : 1.0;
      double nn = 0.0;
      for (int i = 0; i < d; ++i) {
        double v = (double)element(q, q_dtype(dtype), ((size_t)t * H + h) * d + i) * scale;
        qd[(size_t)h * d + i] = v;
        nn += v * v;
      }
      qnorm[h] = sqrt(nn);
    }
    for (int64_t j = 0; j < k_top; ++j) {
      int32_t s = idx[t * k_top + j];
      if (s < 0 || s >= L) continue;
      double g = (double)grad[t * k_top + j];
      const double* ks = kd + (size_t)s * d;
      for (int h = 0; h < H; ++h) {
        double x = 0.0;
        for (int i = 0; i < d; ++i) x += qd[(size_t)h * d + i] * ks[i];
        int amb = fabs(x) <= eps * qnorm[h] * knorm[s];
        double coef = g * (double)w[t * H + h];
        for (int i = 0; i < d; ++i) {
          size_t e = (size_t)s * d + i;
          if (x > 0.0) {
            dk[e] += coef * qd[(size_t)h * d + i];
            if (dk_abs) dk_abs[e] += fabs(coef * qd[(size_t)h * d + i]);
          }
          if (dk_amb && amb) dk_amb[e] += fabs(coef * qd[(size_t)h * d + i]);
        }
      }
    }
  }
  int st = (qd && qnorm) ? ORACLE_OK : ORACLE_NO_MEMORY;
  free(qnorm);
  free(qd);
  free(knorm);
  free(kd);
  if (bad) *bad = nbad;
  return st;
}
