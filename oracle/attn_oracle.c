/*
 * attn_oracle.c -- plain fp64 CPU oracle for scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY (see attn_oracle.h): used by tests, the smoke check
 * and the benchmark's CPU-baseline leg; never by the product path.
 *
 * It is Eq. (1) written out with no blocking, fusion or reordering:
 *   for each (b, h, i):
 *     s_j = scale * sum_t q_{i,t} k_{j,t}          for legal j, else -inf
 *     m   = max_j s_j
 *     w_j = exp(s_j - m)                           (shift-invariance of softmax)
 *     l   = sum_j w_j
 *     o_i = sum_j (w_j / l) v_j
 *     lse = m + ln l
 * Sources: "Attention Is All You Need" (rockcohen.cc) section 3.2 (softmax,
 * shift invariance), section 5.1 (Eq. 1 and the 1/sqrt(d_k) scale), sections
 * 5.3 and 6.3 (-inf at the softmax input, exact-zero weights; the causal mask that
 * makes step-by-step generation legal, used here for the decode mask); vlmlib.cn paper
 * summary, "scaled dot-product attention" and "multi-head attention" (heads are
 * independent attention calls); attention-paper-guide section 03.2 (the
 * four steps: dot products, scale, softmax, weighted sum of V).
 *
 * Inputs are widened exactly to double before any arithmetic. Every sum runs in
 * double in index order. Threads (pthreads) split the query rows; each row is
 * computed by one thread start to finish, so results do not depend on the
 * thread count.
 */
#include "attn_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  const void* q;
  const void* k;
  const void* v;
  int dtype;
  int B, H, n_q, n_k, d_k, d_v;
  double scale;
  int mask_mode;
  const int* key_lens;
  int window;
} problem;

/* Element idx of an input array, widened exactly to double. */
static double elem(const void* base, int dtype, long long idx) {
  if (dtype == ORACLE_F64) return ((const double*)base)[idx];
  if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
  /* bf16 is the upper 16 bits of an IEEE-754 binary32 value */
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Is key j a legal connection for query i of batch b? */
static int legal(const problem* p, int b, int i, int j) {
  if ((p->mask_mode & ORACLE_MASK_CAUSAL) && j > i) return 0;
  if ((p->mask_mode & ORACLE_MASK_KEY_PADDING) && j >= p->key_lens[b]) return 0;
  if ((p->mask_mode & ORACLE_MASK_DECODE) && j > p->key_lens[b] - p->n_q + i) return 0;
  if ((p->mask_mode & ORACLE_MASK_WINDOW) && (j > i + p->window || j < i - p->window)) return 0;
  return 1;
}

/* Scores of query row i of head bh against every key: s[j] = scale * q_i . k_j,
 * or -inf where the connection is illegal. Returns the row maximum. */
static double row_scores(const problem* p, int bh, int i, double* s) {
  int b = bh / p->H;
  long long qoff = ((long long)bh * p->n_q + i) * p->d_k;
  long long koff = (long long)bh * p->n_k * p->d_k;
  double m = -INFINITY;
  for (int j = 0; j < p->n_k; ++j) {
    if (!legal(p, b, i, j)) {
      s[j] = -INFINITY;
      continue;
    }
    double dot = 0.0;
    for (int t = 0; t < p->d_k; ++t)
      dot += elem(p->q, p->dtype, qoff + t) * elem(p->k, p->dtype, koff + (long long)j * p->d_k + t);
    s[j] = p->scale * dot;
    if (s[j] > m) m = s[j];
  }
  return m;
}

/* Turns the scores of one row into softmax weights in place; returns l, the sum
 * of exp(s_j - m). A row with no legal key (m = -inf) becomes all zeros, l = 0. */
static double row_softmax(int n_k, double m, double* s) {
  if (m == -INFINITY) {
    for (int j = 0; j < n_k; ++j) s[j] = 0.0;
    return 0.0;
  }
  double l = 0.0;
  for (int j = 0; j < n_k; ++j) {
    s[j] = exp(s[j] - m); /* exp(-inf) == 0 exactly */
    l += s[j];
  }
  for (int j = 0; j < n_k; ++j) s[j] = s[j] / l;
  return l;
}

/* Output row o_i = sum_j w_j v_j and its log-sum-exp. */
static void attend_row(const problem* p, int bh, int i, double* s, double* o, double* lse) {
  long long voff = (long long)bh * p->n_k * p->d_v;
  double m = row_scores(p, bh, i, s);
  double l = row_softmax(p->n_k, m, s);
  for (int t = 0; t < p->d_v; ++t) o[t] = 0.0;
  for (int j = 0; j < p->n_k; ++j)
    for (int t = 0; t < p->d_v; ++t) o[t] += s[j] * elem(p->v, p->dtype, voff + (long long)j * p->d_v + t);
  if (lse) *lse = (l > 0.0) ? m + log(l) : -INFINITY;
}

typedef struct {
  const problem* p;
  long long n_rows;
  const long long* row_ids; /* NULL: all rows, in order */
  double* out;
  double* lse;
  int tid, n_threads;
  int failed;
} job;

static void* worker(void* arg) {
  job* jb = (job*)arg;
  const problem* p = jb->p;
  double* s = (double*)malloc(sizeof(double) * (size_t)(p->n_k > 0 ? p->n_k : 1));
  if (!s) {
    jb->failed = 1;
    return NULL;
  }
  /* rows are dealt round-robin so that causal rows of different cost spread evenly */
  for (long long r = jb->tid; r < jb->n_rows; r += jb->n_threads) {
    long long id = jb->row_ids ? jb->row_ids[r] : r;
    int bh = (int)(id / p->n_q);
    int i = (int)(id % p->n_q);
    attend_row(p, bh, i, s, jb->out + r * p->d_v, jb->lse ? jb->lse + r : NULL);
  }
  free(s);
  return NULL;
}

static int check(const problem* p) {
  if (!p->q || !p->k) return -1;
  if (p->dtype < ORACLE_F64 || p->dtype > ORACLE_BF16) return -1;
  if (p->B <= 0 || p->H <= 0 || p->n_q <= 0 || p->n_k <= 0 || p->d_k <= 0 || p->d_v < 0) return -1;
  if ((p->mask_mode & ~(ORACLE_MASK_CAUSAL | ORACLE_MASK_KEY_PADDING | ORACLE_MASK_DECODE | ORACLE_MASK_WINDOW)) != 0)
    return -1;
  if ((p->mask_mode & ORACLE_MASK_DECODE) && (p->mask_mode & ORACLE_MASK_WINDOW)) return -1;
  if ((p->mask_mode & ORACLE_MASK_WINDOW) && p->window < 0) return -1;
  if ((p->mask_mode & ORACLE_MASK_CAUSAL) && (p->mask_mode & ORACLE_MASK_DECODE)) return -1;
  if ((p->mask_mode & (ORACLE_MASK_KEY_PADDING | ORACLE_MASK_DECODE)) && !p->key_lens) return -1;
  return 0;
}

static int run(const problem* p, long long n_rows, const long long* row_ids, double* out, double* lse,
               int n_threads) {
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 1024) n_threads = 1024;
  long long total = (long long)p->B * p->H * p->n_q;
  if (row_ids)
    for (long long r = 0; r < n_rows; ++r)
      if (row_ids[r] < 0 || row_ids[r] >= total) return -1;
  job* jobs = (job*)calloc((size_t)n_threads, sizeof(job));
  pthread_t* th = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -1;
  }
  int started = 0;
  for (int t = 0; t < n_threads; ++t) {
    jobs[t] = (job){p, n_rows, row_ids, out, lse, t, n_threads, 0};
    if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) break;
    ++started;
  }
  /* rows of any thread that failed to start are done on this thread */
  for (int t = started; t < n_threads; ++t) worker(&jobs[t]);
  int rc = 0;
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  for (int t = 0; t < n_threads; ++t) rc |= jobs[t].failed;
  free(jobs);
  free(th);
  return rc ? -1 : 0;
}

int oracle_attn(const void* q, const void* k, const void* v, int dtype, int B, int H, int n_q, int n_k,
                int d_k, int d_v, double scale, int mask_mode, const int* key_lens, int window, double* out,
                double* lse, int n_threads) {
  problem p = {q, k, v, dtype, B, H, n_q, n_k, d_k, d_v, scale, mask_mode, key_lens, window};
  if (check(&p) != 0 || !v || !out) return -1;
  return run(&p, (long long)B * H * n_q, NULL, out, lse, n_threads);
}

int oracle_attn_rows(const void* q, const void* k, const void* v, int dtype, int B, int H, int n_q, int n_k,
                     int d_k, int d_v, double scale, int mask_mode, const int* key_lens, int window,
                     long long n_rows, const long long* row_ids, double* out_rows, double* lse_rows,
                     int n_threads) {
  problem p = {q, k, v, dtype, B, H, n_q, n_k, d_k, d_v, scale, mask_mode, key_lens, window};
  if (check(&p) != 0 || !v || !out_rows || !row_ids || n_rows < 0) return -1;
  return run(&p, n_rows, row_ids, out_rows, lse_rows, n_threads);
}

int oracle_attn_weights(const void* q, const void* k, int dtype, int B, int H, int n_q, int n_k, int d_k,
                        double scale, int mask_mode, const int* key_lens, int window, double* weights) {
  problem p = {q, k, NULL, dtype, B, H, n_q, n_k, d_k, 0, scale, mask_mode, key_lens, window};
  if (check(&p) != 0 || !weights) return -1;
  for (int bh = 0; bh < B * H; ++bh)
    for (int i = 0; i < n_q; ++i) {
      double* s = weights + ((long long)bh * n_q + i) * n_k;
      double m = row_scores(&p, bh, i, s);
      row_softmax(n_k, m, s);
    }
  return 0;
}

/* ---------------------------------------------------------------- gradients */
typedef struct {
  const problem* p;
  const void* dout;
  double *dq, *dk, *dv;
  int tid, n_threads;
  int failed;
} bwd_job;

/* Gradients of one head bh, row by row (definitions in attn_oracle.h). */
static void bwd_head(const problem* p, const void* dout, int bh, double* w, double* dp, double* dq, double* dk,
                     double* dv) {
  const long long qoff = (long long)bh * p->n_q * p->d_k, koff = (long long)bh * p->n_k * p->d_k;
  const long long voff = (long long)bh * p->n_k * p->d_v, ooff = (long long)bh * p->n_q * p->d_v;
  for (int i = 0; i < p->n_q; ++i) {
    double m = row_scores(p, bh, i, w);
    row_softmax(p->n_k, m, w); /* w_j = P_ij */
    double sum_pdp = 0.0;
    for (int j = 0; j < p->n_k; ++j) {
      double acc = 0.0;
      for (int t = 0; t < p->d_v; ++t)
        acc += elem(dout, p->dtype, ooff + (long long)i * p->d_v + t) * elem(p->v, p->dtype, voff + (long long)j * p->d_v + t);
      dp[j] = acc;
      sum_pdp += w[j] * acc;
    }
    for (int j = 0; j < p->n_k; ++j) {
      const double ds = w[j] * (dp[j] - sum_pdp);
      for (int t = 0; t < p->d_k; ++t) {
        dq[qoff + (long long)i * p->d_k + t] += p->scale * ds * elem(p->k, p->dtype, koff + (long long)j * p->d_k + t);
        dk[koff + (long long)j * p->d_k + t] += p->scale * ds * elem(p->q, p->dtype, qoff + (long long)i * p->d_k + t);
      }
      for (int t = 0; t < p->d_v; ++t)
        dv[voff + (long long)j * p->d_v + t] += w[j] * elem(dout, p->dtype, ooff + (long long)i * p->d_v + t);
    }
  }
}

static void* bwd_worker(void* arg) {
  bwd_job* jb = (bwd_job*)arg;
  const problem* p = jb->p;
  double* w = (double*)malloc(sizeof(double) * (size_t)p->n_k);
  double* dp = (double*)malloc(sizeof(double) * (size_t)p->n_k);
  if (!w || !dp) {
    jb->failed = 1;
  } else {
    for (int bh = jb->tid; bh < p->B * p->H; bh += jb->n_threads) bwd_head(p, jb->dout, bh, w, dp, jb->dq, jb->dk, jb->dv);
  }
  free(w);
  free(dp);
  return NULL;
}

int oracle_attn_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype, int B, int H, int n_q,
                    int n_k, int d_k, int d_v, double scale, int mask_mode, const int* key_lens, int window, double* dq,
                    double* dk, double* dv, int n_threads) {
  problem p = {q, k, v, dtype, B, H, n_q, n_k, d_k, d_v, scale, mask_mode, key_lens, window};
  if (check(&p) != 0 || !v || !dout || !dq || !dk || !dv) return -1;
  memset(dq, 0, sizeof(double) * (size_t)B * H * n_q * d_k);
  memset(dk, 0, sizeof(double) * (size_t)B * H * n_k * d_k);
  memset(dv, 0, sizeof(double) * (size_t)B * H * n_k * d_v);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > B * H) n_threads = B * H;
  bwd_job* jobs = (bwd_job*)calloc((size_t)n_threads, sizeof(bwd_job));
  pthread_t* th = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -1;
  }
  int started = 0;
  for (int t = 0; t < n_threads; ++t) {
    jobs[t] = (bwd_job){&p, dout, dq, dk, dv, t, n_threads, 0};
    if (pthread_create(&th[t], NULL, bwd_worker, &jobs[t]) != 0) break;
    ++started;
  }
  for (int t = started; t < n_threads; ++t) bwd_worker(&jobs[t]);
  int rc = 0;
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  for (int t = 0; t < n_threads; ++t) rc |= jobs[t].failed;
  free(jobs);
  free(th);
  return rc ? -1 : 0;
}

/* ---------------------------------------------------------------- multi-head attention */
/* x [B, n, d_in] times the head-i columns of w [d_in, H*d] (+ bias), written head-split
 * as out [B, H, n, d]. */
static void project_heads(const void* x, const void* w, const void* bias, int dtype, int B, int n, int d_in, int H,
                          int d, double* out) {
  const long long wcols = (long long)H * d;
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < n; ++i) {
      const long long xrow = ((long long)b * n + i) * d_in;
      for (int h = 0; h < H; ++h)
        for (int t = 0; t < d; ++t) {
          const long long col = (long long)h * d + t;
          double acc = bias ? elem(bias, dtype, col) : 0.0;
          for (int c = 0; c < d_in; ++c) acc += elem(x, dtype, xrow + c) * elem(w, dtype, (long long)c * wcols + col);
          out[(((long long)b * H + h) * n + i) * d + t] = acc;
        }
    }
}

int oracle_mha(const void* x_q, const void* x_kv, int dtype, const void* w_q, const void* b_q, const void* w_k,
               const void* b_k, const void* w_v, const void* b_v, const void* w_o, const void* b_o, int B, int n_q,
               int n_k, int d_model, int H, int d_k, int d_v, double scale, int mask_mode, const int* key_lens,
               double* y, int n_threads) {
  if (!x_q || !x_kv || !w_q || !w_k || !w_v || !w_o || !y) return -1;
  if (dtype < ORACLE_F64 || dtype > ORACLE_BF16) return -1;
  if (B <= 0 || n_q <= 0 || n_k <= 0 || d_model <= 0 || H <= 0 || d_k <= 0 || d_v <= 0) return -1;
  if (mask_mode & (ORACLE_MASK_DECODE | ORACLE_MASK_WINDOW)) return -1;
  const size_t nq = (size_t)B * H * n_q, nk = (size_t)B * H * n_k;
  double* qh = (double*)malloc(nq * d_k * sizeof(double));
  double* kh = (double*)malloc(nk * d_k * sizeof(double));
  double* vh = (double*)malloc(nk * d_v * sizeof(double));
  double* oh = (double*)malloc(nq * d_v * sizeof(double));
  int rc = -1;
  if (qh && kh && vh && oh) {
    /* the three linear projections, split into heads: head i uses columns i*d_k.. of W^Q */
    project_heads(x_q, w_q, b_q, dtype, B, n_q, d_model, H, d_k, qh);
    project_heads(x_kv, w_k, b_k, dtype, B, n_k, d_model, H, d_k, kh);
    project_heads(x_kv, w_v, b_v, dtype, B, n_k, d_model, H, d_v, vh);
    /* scaled dot-product attention per head */
    rc = oracle_attn(qh, kh, vh, ORACLE_F64, B, H, n_q, n_k, d_k, d_v, scale, mask_mode, key_lens, 0, oh, NULL,
                     n_threads);
    if (rc == 0) {
      /* concatenate the heads along the feature axis (head h fills columns h*d_v..) and
       * apply the output projection W^O [H*d_v, d_model] */
      for (int b = 0; b < B; ++b)
        for (int i = 0; i < n_q; ++i)
          for (int c = 0; c < d_model; ++c) {
            double acc = b_o ? elem(b_o, dtype, c) : 0.0;
            for (int h = 0; h < H; ++h)
              for (int t = 0; t < d_v; ++t)
                acc += oh[(((long long)b * H + h) * n_q + i) * d_v + t] *
                       elem(w_o, dtype, ((long long)h * d_v + t) * d_model + c);
            y[((long long)b * n_q + i) * d_model + c] = acc;
          }
    }
  }
  free(qh);
  free(kh);
  free(vh);
  free(oh);
  return rc;
}

int oracle_linear(const void* x, const void* w, const void* bias, int dtype, int M, int N, int K, double* y) {
  if (!x || !w || !y || M <= 0 || N <= 0 || K <= 0) return -1;
  if (dtype < ORACLE_F64 || dtype > ORACLE_BF16) return -1;
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      double acc = bias ? elem(bias, dtype, n) : 0.0;
      for (int k = 0; k < K; ++k) acc += elem(x, dtype, (long long)m * K + k) * elem(w, dtype, (long long)k * N + n);
      y[(long long)m * N + n] = acc;
    }
  return 0;
}
