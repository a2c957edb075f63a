/*
 * vattn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, double-precision CPU oracle for non-causal head-major
 * attention, out = softmax(Q K^T) V, as computed by the WGSL shader
 * "vision_attention_flash_sub_hpd_f16.wgsl" (rullama 0.1.0).  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may call it;
 * the product path never does.
 *
 * What it follows on that page:
 *   - buffer layout: head-major (HPD); element (h, n, d) of q, k, v and out
 *     sits at h*n_patches*head_dim + n*head_dim + d ("Buffer layout =
 *     head-major", the head_base / q_off / out_off arithmetic of main()).
 *     A batch is folded into the head index (b*n_heads + h): contiguous
 *     [batch, n_heads, n_patches, head_dim] is the same memory as
 *     [batch*n_heads, n_patches, head_dim].
 *   - score: s_j = sum_d q[i,d] * k[j,d], with no 1/sqrt(head_dim) factor
 *     (the score loop applies none; the caller pre-scales q).
 *   - normalisation: the running (m, l, o) online softmax of the tile loop,
 *     finished by out = o / l.  Online softmax is an exact rewrite of the
 *     plain softmax, so this oracle writes out the plain definition instead,
 *     in three passes per query row:
 *        pass 1: s_j for every key j (d ascending), m = max_j s_j
 *        pass 2: p_j = exp(s_j - m), l = sum_j p_j (j ascending)
 *        pass 3: out[i,d] = (sum_j p_j v[j,d]) / l (j ascending)
 *     The f16 staging of the shader is its approximation and is not
 *     reproduced: inputs are the exact f32 values widened to double.
 *
 * Threads split the query rows; each row is computed by one thread in a
 * fixed order, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define VATTN_ORACLE_OK 0
#define VATTN_ORACLE_EINVAL 1
#define VATTN_ORACLE_ENOMEM 2

/* One query row: q_row[D], k_head/v_head [N, D] (one head), out_row[D]. */
static void oracle_row(const float *q_row, const float *k_head,
                       const float *v_head, int64_t n_patches,
                       int64_t head_dim, double *p /* [n_patches] */,
                       double *out_row) {
  /* pass 1: scores and their maximum */
  double m = -INFINITY;
  for (int64_t j = 0; j < n_patches; ++j) {
    const float *k_row = k_head + j * head_dim;
    double s = 0.0;
    for (int64_t d = 0; d < head_dim; ++d)
      s += (double)q_row[d] * (double)k_row[d];
    p[j] = s;
    if (s > m) m = s;
  }
  /* pass 2: exponentials relative to the maximum and their sum */
  double l = 0.0;
  for (int64_t j = 0; j < n_patches; ++j) {
    p[j] = exp(p[j] - m);
    l += p[j];
  }
  /* pass 3: weighted sum of value rows, divided by the sum */
  for (int64_t d = 0; d < head_dim; ++d) out_row[d] = 0.0;
  for (int64_t j = 0; j < n_patches; ++j) {
    const float *v_row = v_head + j * head_dim;
    const double w = p[j];
    for (int64_t d = 0; d < head_dim; ++d) out_row[d] += w * (double)v_row[d];
  }
  for (int64_t d = 0; d < head_dim; ++d) out_row[d] /= l;
}

typedef struct {
  const float *q, *k, *v;
  int64_t n_patches, head_dim;
  const int64_t *rows; /* NULL: rows [first, last) of the full tensor */
  int64_t first, last;
  double *out;
  int status;
} oracle_job;

static void *oracle_worker(void *arg) {
  oracle_job *job = (oracle_job *)arg;
  const int64_t N = job->n_patches, D = job->head_dim;
  double *p = (double *)malloc((size_t)N * sizeof(double));
  if (!p) {
    job->status = VATTN_ORACLE_ENOMEM;
    return NULL;
  }
  for (int64_t r = job->first; r < job->last; ++r) {
    /* flat row index = bh * N + i */
    const int64_t flat = job->rows ? job->rows[r] : r;
    const int64_t bh = flat / N;
    const float *k_head = job->k + bh * N * D;
    const float *v_head = job->v + bh * N * D;
    oracle_row(job->q + flat * D, k_head, v_head, N, D, p,
               job->out + r * D);
  }
  free(p);
  job->status = VATTN_ORACLE_OK;
  return NULL;
}

static int run_jobs(const float *q, const float *k, const float *v,
                    int64_t n_patches, int64_t head_dim, const int64_t *rows,
                    int64_t n_rows, double *out, int threads) {
  if (threads < 1) threads = 1;
  if ((int64_t)threads > n_rows) threads = (int)(n_rows > 0 ? n_rows : 1);
  oracle_job *jobs = (oracle_job *)calloc((size_t)threads, sizeof(oracle_job));
  pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
  int *started = (int *)calloc((size_t)threads, sizeof(int));
  if (!jobs || !tids || !started) {
    free(jobs);
    free(tids);
    free(started);
    return VATTN_ORACLE_ENOMEM;
  }
  int status = VATTN_ORACLE_OK;
  for (int t = 0; t < threads; ++t) {
    jobs[t].q = q;
    jobs[t].k = k;
    jobs[t].v = v;
    jobs[t].n_patches = n_patches;
    jobs[t].head_dim = head_dim;
    jobs[t].rows = rows;
    jobs[t].first = n_rows * t / threads;
    jobs[t].last = n_rows * (t + 1) / threads;
    jobs[t].out = out;
    jobs[t].status = VATTN_ORACLE_OK;
    if (t == threads - 1) {
      oracle_worker(&jobs[t]); /* the calling thread takes the last share */
    } else if (pthread_create(&tids[t], NULL, oracle_worker, &jobs[t]) == 0) {
      started[t] = 1;
    } else {
      oracle_worker(&jobs[t]);
    }
  }
  for (int t = 0; t < threads; ++t) {
    if (started[t]) pthread_join(tids[t], NULL);
    if (jobs[t].status != VATTN_ORACLE_OK) status = jobs[t].status;
  }
  free(jobs);
  free(tids);
  free(started);
  return status;
}

/*
 * Full tensor: q, k, v are [batch, n_heads, n_patches, head_dim] f32,
 * out is the same shape in f64.  Empty problems (any size 0) are no-ops.
 */
int vattn_oracle_forward(const float *q, const float *k, const float *v,
                         double *out, int64_t batch, int64_t n_heads,
                         int64_t n_patches, int64_t head_dim, int threads) {
  if (batch < 0 || n_heads < 0 || n_patches < 0 || head_dim < 0)
    return VATTN_ORACLE_EINVAL;
  const int64_t n_rows = batch * n_heads * n_patches;
  if (n_rows == 0 || head_dim == 0) return VATTN_ORACLE_OK;
  if (!q || !k || !v || !out) return VATTN_ORACLE_EINVAL;
  return run_jobs(q, k, v, n_patches, head_dim, NULL, n_rows, out, threads);
}

/*
 * Selected rows only: rows[r] is a flat query-row index bh*n_patches + i
 * into q (bh < n_bh); out is [n_rows, head_dim] f64, row r for rows[r].
 */
int vattn_oracle_rows(const float *q, const float *k, const float *v,
                      int64_t n_bh, int64_t n_patches, int64_t head_dim,
                      const int64_t *rows, int64_t n_rows, double *out,
                      int threads) {
  if (n_bh < 0 || n_patches < 0 || head_dim < 0 || n_rows < 0)
    return VATTN_ORACLE_EINVAL;
  if (n_rows == 0 || head_dim == 0) return VATTN_ORACLE_OK;
  if (!q || !k || !v || !out || !rows) return VATTN_ORACLE_EINVAL;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= n_bh * n_patches) return VATTN_ORACLE_EINVAL;
  return run_jobs(q, k, v, n_patches, head_dim, rows, n_rows, out, threads);
}
