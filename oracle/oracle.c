/*
 * oracle.c -- fp64 CPU oracle for row-wise softmax.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference leg are the only callers.  The CUDA
 * library never calls, links or includes anything here, and nothing here is
 * taken from the CUDA library: the two share no code.
 *
 * What it computes, in double precision, written as the plain definitions:
 *
 *  oracle_softmax_rows -- the three-pass safe softmax of a row
 *      ("5.2 CUDA Online Softmax 实现优化", §1.1; "Softmax 数值稳定性与
 *       IO-Aware Attention", §三):
 *          pass 1:  m   = max_j x_j
 *          pass 2:  d   = sum_j exp(x_j - m)
 *          pass 3:  y_j = exp(x_j - m) / d
 *      and the log-sum-exp  LSE = m + log(d)
 *      ("从原始Softmax到在线Softmax", section "softmax形式推导").
 *
 *  Every row function takes the softmax of z = scale * x (scale > 0; z is exact
 *  in double), which is x itself for scale 1.
 *
 *  oracle_log_softmax_rows -- the log of the softmax, as the page's
 *      log_probs = x - max - log(sum_j exp(x_j - max))
 *      ("从原始Softmax到在线Softmax", section "softmax实际代码实现").
 *
 *  oracle_cross_entropy_rows -- the per-row cross-entropy loss of the same
 *      section's cross_entropy_loss, -log_probs[r, label_r], before its mean
 *      over rows (worked example "交叉熵损失计算": 0.4170).
 *
 *  oracle_online_state -- the element-by-element (m, d) recurrence
 *      ("5.2 CUDA Online Softmax 实现优化", §2.1):
 *          m_{k+1} = max(m_k, x_k)
 *          d_{k+1} = d_k * exp(m_k - m_{k+1}) + exp(x_k - m_{k+1})
 *
 *  oracle_merge_state -- the merge of two partial states
 *      ("5.2 CUDA Online Softmax 实现优化", §4.1; "Softmax 数值稳定性与
 *       IO-Aware Attention", §4.1):
 *          m = max(m_a, m_b)
 *          d = d_a * exp(m_a - m) + d_b * exp(m_b - m)
 *
 * Readings where the pages are silent:
 *  - exp(a - b) is taken as 0 whenever a = -inf.  So the empty state
 *    (-inf, 0) is the identity of the merge and of the recurrence, as in the
 *    worked merge of "从原始Softmax到在线Softmax" (section "手推小例子": the
 *    first merge uses scale_old = 0 for m_old = -inf), and no -inf - (-inf)
 *    is ever evaluated.
 *  - A row whose entries are all -inf has y = 0, m = -inf, d = 0, LSE = -inf.
 *  - bf16 and fp16 inputs are widened exactly (bf16 -> fp32 -> fp64; fp16 -> fp64).
 *  - log softmax of an all -inf row is -inf everywhere (log 0).
 *  - Cross entropy: a negative label marks a row to ignore (loss 0); a label
 *    >= N gives NaN.  A row whose labelled entry is -inf has loss +inf
 *    (-log 0); an all -inf row gives -inf - (-inf) = NaN.
 *
 * Rows are independent, so they are spread over POSIX threads; inside a row
 * the three passes run in plain index order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F16 2

/* Element i of a row-major matrix of the given dtype, widened exactly (the C compiler's
 * IEEE binary16 type for fp16). */
static double load_elem(const void* x, int dtype, int64_t i) {
  if (dtype == ORACLE_F32) return (double)((const float*)x)[i];
  if (dtype == ORACLE_F16) {
    _Float16 h;
    memcpy(&h, (const uint16_t*)x + i, sizeof h);
    return (double)h;
  }
  uint32_t bits = (uint32_t)((const uint16_t*)x)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* exp(a - b), with exp(-inf - b) := 0 (the empty-state reading above). */
static double scaled_exp(double a, double b) {
  if (a == -INFINITY) return 0.0;
  return exp(a - b);
}

/* The softmax input z = scale * x (exact in double: a 24-bit scale times a value of at most 24
 * significant bits). */
static double load_z(const void* x, int dtype, int64_t i, double scale) {
  return scale * load_elem(x, dtype, i);
}

/* Three-pass safe softmax of row `row` of z = scale * x; y may be NULL (state only). */
static void softmax_one_row(const void* x, int dtype, int64_t N, int64_t row, double scale,
                            double* y, double* m_out, double* d_out,
                            double* lse_out) {
  const int64_t base = row * N;

  /* pass 1: the row maximum */
  double m = -INFINITY;
  for (int64_t j = 0; j < N; ++j) {
    double v = load_z(x, dtype, base + j, scale);
    if (v > m) m = v;
  }

  /* pass 2: the denominator */
  double d = 0.0;
  for (int64_t j = 0; j < N; ++j) d += scaled_exp(load_z(x, dtype, base + j, scale), m);

  /* pass 3: normalise */
  if (y) {
    for (int64_t j = 0; j < N; ++j) {
      y[j] = (m == -INFINITY) ? 0.0 : scaled_exp(load_z(x, dtype, base + j, scale), m) / d;
    }
  }
  if (m_out) *m_out = m;
  if (d_out) *d_out = d;
  if (lse_out) *lse_out = (m == -INFINITY) ? -INFINITY : m + log(d);
}

typedef struct {
  const void* x;
  int dtype;
  int64_t N;
  const int64_t* rows;
  int64_t nrows;
  double *y, *m, *d, *lse;
  int64_t begin, end; /* slice of [0, nrows) handled by this thread */
  double scale;
} oracle_job;

static void* oracle_worker(void* arg) {
  oracle_job* job = (oracle_job*)arg;
  for (int64_t i = job->begin; i < job->end; ++i) {
    int64_t row = job->rows ? job->rows[i] : i;
    softmax_one_row(job->x, job->dtype, job->N, row, job->scale,
                    job->y ? job->y + i * job->N : NULL,
                    job->m ? job->m + i : NULL, job->d ? job->d + i : NULL,
                    job->lse ? job->lse + i : NULL);
  }
  return NULL;
}

/*
 * Softmax of z = scale * x for selected rows of a row-major matrix x (dtype
 * ORACLE_F32, ORACLE_BF16 or ORACLE_F16, N columns); scale > 0.  rows[i] is the i-th row to compute, or rows ==
 * NULL for rows 0..nrows-1.  Outputs are indexed by i: y is nrows x N,
 * m / d / lse have nrows entries; each output may be NULL.  Returns 0, or -1
 * on a bad argument.
 */
int oracle_softmax_rows_scaled(const void* x, int dtype, int64_t N,
                               const int64_t* rows, int64_t nrows, double scale,
                               double* y, double* m, double* d, double* lse,
                               int nthreads) {
  if (!x || N < 1 || nrows < 0) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
  if (nrows == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nrows) nthreads = (int)nrows;

  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
  if (!tids || !jobs) {
    free(tids);
    free(jobs);
    return -1;
  }
  for (int t = 0; t < nthreads; ++t) {
    oracle_job job = {x, dtype, N, rows, nrows, y, m, d, lse,
                      nrows * t / nthreads, nrows * (t + 1) / nthreads, scale};
    jobs[t] = job;
    if (t == 0) continue; /* the calling thread takes slice 0 */
    if (pthread_create(&tids[t], NULL, oracle_worker, &jobs[t]) != 0) {
      oracle_worker(&jobs[t]); /* no thread available: do it inline */
      tids[t] = (pthread_t)0;
    }
  }
  oracle_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (tids[t] != (pthread_t)0) pthread_join(tids[t], NULL);
  free(tids);
  free(jobs);
  return 0;
}

/* The softmax of x itself (scale 1). */
int oracle_softmax_rows(const void* x, int dtype, int64_t N, const int64_t* rows, int64_t nrows,
                        double* y, double* m, double* d, double* lse, int nthreads) {
  return oracle_softmax_rows_scaled(x, dtype, N, rows, nrows, 1.0, y, m, d, lse, nthreads);
}

/* The row's m and d (passes 1 and 2 of the three-pass softmax above). */
static void row_max_and_sum(const void* x, int dtype, int64_t N, int64_t row, double scale, double* m_out,
                            double* d_out) {
  const int64_t base = row * N;
  double m = -INFINITY;
  for (int64_t j = 0; j < N; ++j) {
    double v = load_z(x, dtype, base + j, scale);
    if (v > m) m = v;
  }
  double d = 0.0;
  for (int64_t j = 0; j < N; ++j) d += scaled_exp(load_z(x, dtype, base + j, scale), m);
  *m_out = m;
  *d_out = d;
}

typedef struct {
  const void* x;
  int dtype;
  int64_t N;
  const int64_t* rows;   /* log softmax: selected rows, or NULL */
  const int64_t* labels; /* cross entropy: one label per row */
  double* out;           /* log softmax: nrows x N; cross entropy: nrows */
  int64_t begin, end;
  double scale;
} oracle_log_job;

static void* oracle_log_worker(void* arg) {
  oracle_log_job* job = (oracle_log_job*)arg;
  for (int64_t i = job->begin; i < job->end; ++i) {
    int64_t row = job->rows ? job->rows[i] : i;
    double m, d;
    row_max_and_sum(job->x, job->dtype, job->N, row, job->scale, &m, &d);
    /* log_probs = x - max - log(sum_exp); all -inf row: -inf */
    double log_d = (m == -INFINITY) ? INFINITY : log(d);
    double shift = (m == -INFINITY) ? 0.0 : m;
    if (!job->labels) {
      double* ly = job->out + i * job->N;
      for (int64_t j = 0; j < job->N; ++j) ly[j] = load_z(job->x, job->dtype, row * job->N + j, job->scale) - shift - log_d;
    } else {
      int64_t label = job->labels[i];
      double loss;
      if (label < 0) {
        loss = 0.0;
      } else if (label >= job->N) {
        loss = NAN;
      } else {
        double xl = load_z(job->x, job->dtype, row * job->N + label, job->scale);
        loss = (m == -INFINITY) ? NAN : -(xl - m - log(d));
      }
      job->out[i] = loss;
    }
  }
  return NULL;
}

static int run_log_jobs(oracle_log_job proto, int64_t nrows, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nrows) nthreads = (int)nrows;
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  oracle_log_job* jobs = (oracle_log_job*)calloc((size_t)nthreads, sizeof(oracle_log_job));
  if (!tids || !jobs) {
    free(tids);
    free(jobs);
    return -1;
  }
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].begin = nrows * t / nthreads;
    jobs[t].end = nrows * (t + 1) / nthreads;
    if (t == 0) continue;
    if (pthread_create(&tids[t], NULL, oracle_log_worker, &jobs[t]) != 0) {
      oracle_log_worker(&jobs[t]);
      tids[t] = (pthread_t)0;
    }
  }
  oracle_log_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (tids[t] != (pthread_t)0) pthread_join(tids[t], NULL);
  free(tids);
  free(jobs);
  return 0;
}

/*
 * Log softmax of z = scale * x for selected rows (rows == NULL: rows
 * 0..nrows-1) into ly (nrows x N).  Returns 0, or -1 on a bad argument.
 */
int oracle_log_softmax_rows(const void* x, int dtype, int64_t N, const int64_t* rows, int64_t nrows,
                            double scale, double* ly, int nthreads) {
  if (!x || !ly || N < 1 || nrows < 0 || !(scale > 0.0)) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
  if (nrows == 0) return 0;
  oracle_log_job proto = {x, dtype, N, rows, NULL, ly, 0, 0, scale};
  return run_log_jobs(proto, nrows, nthreads);
}

/*
 * Cross-entropy loss of rows 0..M-1 against labels[0..M) into loss[0..M).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_cross_entropy_rows(const void* x, int dtype, int64_t N, const int64_t* labels, int64_t M,
                              double* loss, int nthreads) {
  if (!x || !labels || !loss || N < 1 || M < 0) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
  if (M == 0) return 0;
  oracle_log_job proto = {x, dtype, N, NULL, labels, loss, 0, 0, 1.0};
  return run_log_jobs(proto, M, nthreads);
}

/*
 * The online recurrence over xs[0..n), one element at a time, starting from
 * the empty state (m, d) = (-inf, 0).
 */
void oracle_online_state(const double* xs, int64_t n, double* m_out, double* d_out) {
  double m = -INFINITY, d = 0.0;
  for (int64_t k = 0; k < n; ++k) {
    double m_new = xs[k] > m ? xs[k] : m;
    if (m_new == -INFINITY) continue; /* -inf element into an empty state: still empty */
    d = d * scaled_exp(m, m_new) + scaled_exp(xs[k], m_new);
    m = m_new;
  }
  *m_out = m;
  *d_out = d;
}

/* Merge of two partial states (m_a, d_a) and (m_b, d_b). */
void oracle_merge_state(double m_a, double d_a, double m_b, double d_b,
                        double* m_out, double* d_out) {
  double m = m_a > m_b ? m_a : m_b;
  if (m == -INFINITY) {
    *m_out = -INFINITY;
    *d_out = 0.0;
    return;
  }
  *m_out = m;
  *d_out = d_a * scaled_exp(m_a, m) + d_b * scaled_exp(m_b, m);
}

/*
 * Attention forward, the plain definition ("从原始Softmax到在线Softmax", worked example
 * "标准 Attention 中的 Softmax": S = Q K^T / sqrt(d), row-wise softmax, O = P V), in double:
 * for the selected query rows, with q, k, v row-major [BH][S][d] of dtype (ORACLE_F32,
 * ORACLE_BF16 or ORACLE_F16) and row i of head h attending keys j < Sk (causal: j <= i + Sk - Sq,
 * the last query row sees every key):
 *     s_j = scale * sum_c q[h][i][c] k[h][j][c],  m = max_j s_j,  l = sum_j e^(s_j - m)
 *     o = sum_j e^(s_j - m) v[h][j] / l,  lse = m + log l.
 * sel[2 * t] = head, sel[2 * t + 1] = query row of the t-th selected row; o is nsel x d, lse has
 * nsel entries.  A row that sees no key gets o = 0, lse = -inf.  Returns 0, or -1 on a bad argument.
 */
typedef struct {
  const void *q, *k, *v;
  int dtype;
  int64_t Sq, Sk, d;
  double scale;
  int causal;
  const int64_t* sel;
  double *o, *lse;
  int64_t begin, end;
} oracle_attn_job;

static void* oracle_attn_worker(void* arg) {
  oracle_attn_job* jb = (oracle_attn_job*)arg;
  double* s = (double*)malloc(sizeof(double) * (size_t)(jb->Sk > 0 ? jb->Sk : 1));
  if (!s) return NULL;
  for (int64_t t = jb->begin; t < jb->end; ++t) {
    const int64_t h = jb->sel[2 * t], i = jb->sel[2 * t + 1];
    int64_t nk = jb->Sk;
    if (jb->causal) {
      nk = i + jb->Sk - jb->Sq + 1;
      if (nk < 0) nk = 0;
      if (nk > jb->Sk) nk = jb->Sk;
    }
    const int64_t qb = (h * jb->Sq + i) * jb->d;
    double m = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) {
      const int64_t kb = (h * jb->Sk + j) * jb->d;
      double dot = 0.0;
      for (int64_t c = 0; c < jb->d; ++c) dot += load_elem(jb->q, jb->dtype, qb + c) * load_elem(jb->k, jb->dtype, kb + c);
      s[j] = jb->scale * dot;
      if (s[j] > m) m = s[j];
    }
    double* o = jb->o + t * jb->d;
    for (int64_t c = 0; c < jb->d; ++c) o[c] = 0.0;
    double l = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
      const double p = exp(s[j] - m);
      l += p;
      const int64_t vb = (h * jb->Sk + j) * jb->d;
      for (int64_t c = 0; c < jb->d; ++c) o[c] += p * load_elem(jb->v, jb->dtype, vb + c);
    }
    if (nk > 0)
      for (int64_t c = 0; c < jb->d; ++c) o[c] /= l;
    jb->lse[t] = nk > 0 ? m + log(l) : -INFINITY;
  }
  free(s);
  return NULL;
}

int oracle_attention_rows(const void* q, const void* k, const void* v, int dtype, int64_t Sq, int64_t Sk,
                          int64_t d, double scale, int causal, const int64_t* sel, int64_t nsel, double* o,
                          double* lse, int nthreads) {
  if (!q || !k || !v || !sel || !o || !lse || Sq < 1 || Sk < 1 || d < 1 || nsel < 0) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
  if (nsel == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nsel) nthreads = (int)nsel;
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  oracle_attn_job* jobs = (oracle_attn_job*)calloc((size_t)nthreads, sizeof(oracle_attn_job));
  if (!tids || !jobs) {
    free(tids);
    free(jobs);
    return -1;
  }
  for (int t = 0; t < nthreads; ++t) {
    oracle_attn_job jb = {q, k, v, dtype, Sq, Sk, d, scale, causal, sel, o, lse,
                          nsel * t / nthreads, nsel * (t + 1) / nthreads};
    jobs[t] = jb;
    if (t == 0) continue;
    if (pthread_create(&tids[t], NULL, oracle_attn_worker, &jobs[t]) != 0) {
      oracle_attn_worker(&jobs[t]);
      tids[t] = (pthread_t)0;
    }
  }
  oracle_attn_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (tids[t] != (pthread_t)0) pthread_join(tids[t], NULL);
  free(tids);
  free(jobs);
  return 0;
}

/*
 * The block recurrence of the same page ("从原始Softmax到在线Softmax", the online-softmax form
 * of the blocked computation): for one query, scores s[0..n) and value rows v[n][d], blocks of
 * `block` keys, starting from m = -inf, l = 0, o~ = 0:
 *     m' = max(m, max of the block)
 *     o~ = e^(m - m') o~ + sum_{k in block} e^(s_k - m') v_k
 *     l  = e^(m - m') l  + sum_{k in block} e^(s_k - m')
 * then o = o~ / l (written to o[0..d)).  e^(-inf - m') is taken as 0.
 */
void oracle_attention_online(const double* s, const double* v, int64_t n, int64_t d, int64_t block, double* o) {
  double m = -INFINITY, l = 0.0;
  for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
  if (block < 1) block = 1;
  for (int64_t b0 = 0; b0 < n; b0 += block) {
    const int64_t b1 = b0 + block < n ? b0 + block : n;
    double mb = -INFINITY;
    for (int64_t k = b0; k < b1; ++k)
      if (s[k] > mb) mb = s[k];
    const double m_new = mb > m ? mb : m;
    if (m_new == -INFINITY) continue;
    const double corr = scaled_exp(m, m_new);
    l *= corr;
    for (int64_t c = 0; c < d; ++c) o[c] *= corr;
    for (int64_t k = b0; k < b1; ++k) {
      const double p = scaled_exp(s[k], m_new);
      l += p;
      for (int64_t c = 0; c < d; ++c) o[c] += p * v[k * d + c];
    }
    m = m_new;
  }
  if (l > 0.0)
    for (int64_t c = 0; c < d; ++c) o[c] /= l;
}
