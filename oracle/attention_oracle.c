/*
 * attention_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * The plain CPU oracle for the attention forward pass that consumes the GEMM
 * pipeline: per batch b and head h, O = softmax(scale * Q K^T, causal mask) V.
 * Only tests/, the smoke check and the CPU-baseline leg of the benchmark use
 * it; the product path never links or calls it and shares no code with it.
 *
 * What it computes ("TileLang: a tile language one level below Triton",
 * section "FlashAttention: online softmax as tile code"):
 *   - Q, K, V and O are [batch, seq, heads, dim] arrays (dim contiguous);
 *   - the scores of query i are s_j = scale * sum_d Q[i][d] * K[j][d], with
 *     scale = 1/sqrt(dim) by default (the section folds log2(e) into it only
 *     to use exp2; exp2(x * log2 e) = exp(x), so the definition uses exp);
 *   - with the causal mask query i sees the keys j <= i (the section's
 *     condition: query index >= key index keeps the score);
 *   - the running maximum, the rescaling of the accumulator and the final
 *     division by the row sum of the online softmax are exact algebra, so the
 *     tiled pass reaches the plain softmax:
 *
 *       m       = max_j s_j                                   (visible j)
 *       p_j     = exp(s_j - m) / sum_j' exp(s_j' - m)
 *       out[d]  = sum_j p_j * V[j][d]
 *       bound[d]= sum_j p_j * |V[j][d]|                        (fp64)
 *
 * The inputs are the fp16/bf16 arrays the GPU sees, widened exactly to fp64 by
 * the caller. Loops run in increasing j and d, built with -ffp-contract=off and
 * no fast-math. (b, row, h) triples are split across POSIX threads; each is
 * still one sequential computation, so the thread count never changes a value.
 *
 * ORACLE_PLANT (test builds only) compiles a deliberate mistake so the pinning
 * tests can show each kind is caught:
 *   11 = strict causal mask (j < i), 12 = scale ignored, 13 = no division by
 *   the row sum, 14 = Q and K exchanged in the score (s_j = Q[j] . K[i]),
 *   15 = V read from head 0 for every head.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

typedef struct {
  const double *Q, *K, *V;
  int64_t batch, seq, heads, dim;
  double scale;
  int causal;
  const int64_t *rows; /* query positions, NULL = 0 .. n_rows-1 */
  int64_t n_rows;
  double *out, *bound; /* [batch][n_rows][heads][dim] */
  int64_t item_begin, item_end;
  int status;
} oracle_attn_job;

/* element [b][s][h][d] of a [batch, seq, heads, dim] array */
static inline int64_t bshd(const oracle_attn_job *j, int64_t b, int64_t s, int64_t h) {
  return ((b * j->seq + s) * j->heads + h) * j->dim;
}

static void oracle_attn_items(oracle_attn_job *job) {
  const int64_t D = job->dim;
  double *score = (double *)malloc((size_t)(job->seq > 0 ? job->seq : 1) * sizeof(double));
  if (!score) {
    job->status = -1;
    return;
  }
  for (int64_t it = job->item_begin; it < job->item_end; ++it) {
    /* item = (b * n_rows + r) * heads + h */
    const int64_t h = it % job->heads;
    const int64_t r = (it / job->heads) % job->n_rows;
    const int64_t b = it / (job->heads * job->n_rows);
    const int64_t i = job->rows ? job->rows[r] : r;
    double *o = job->out + ((b * job->n_rows + r) * job->heads + h) * D;
    double *ob = job->bound + ((b * job->n_rows + r) * job->heads + h) * D;
#if ORACLE_PLANT == 11
    const int64_t visible = job->causal ? i : job->seq;
#else
    const int64_t visible = job->causal ? i + 1 : job->seq; /* keys 0 .. visible-1 */
#endif
#if ORACLE_PLANT == 12
    const double scale = 1.0;
#else
    const double scale = job->scale;
#endif
    double m = -INFINITY;
    for (int64_t j = 0; j < visible; ++j) {
#if ORACLE_PLANT == 14
      const double *q = job->Q + bshd(job, b, j, h);
      const double *k = job->K + bshd(job, b, i, h);
#else
      const double *q = job->Q + bshd(job, b, i, h);
      const double *k = job->K + bshd(job, b, j, h);
#endif
      double dot = 0.0;
      for (int64_t d = 0; d < D; ++d) dot += q[d] * k[d];
      score[j] = scale * dot;
      if (score[j] > m) m = score[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < visible; ++j) {
      score[j] = exp(score[j] - m);
      denom += score[j];
    }
#if ORACLE_PLANT == 13
    denom = 1.0;
#endif
    for (int64_t d = 0; d < D; ++d) {
      o[d] = 0.0;
      ob[d] = 0.0;
    }
    for (int64_t j = 0; j < visible; ++j) {
      const double p = score[j] / denom;
#if ORACLE_PLANT == 15
      const double *v = job->V + bshd(job, b, j, 0);
#else
      const double *v = job->V + bshd(job, b, j, h);
#endif
      for (int64_t d = 0; d < D; ++d) {
        o[d] += p * v[d];
        ob[d] += p * fabs(v[d]);
      }
    }
  }
  free(score);
}

static void *oracle_attn_thread(void *arg) {
  oracle_attn_items((oracle_attn_job *)arg);
  return NULL;
}

/*
 * oracle_attention_f64: out and bound, [batch][n_rows][heads][dim] fp64, for
 * the query positions rows[0 .. n_rows-1] (rows == NULL: positions 0 ..
 * n_rows-1) of every batch and head. Q, K, V are [batch][seq][heads][dim] fp64
 * host arrays owned by the caller. causal != 0 applies the causal mask.
 * nthreads <= 0 means one thread. Returns 0, or -1 on bad sizes, a row outside
 * 0 .. seq-1, or an allocation / thread failure.
 */
int oracle_attention_f64(const double *Q, const double *K, const double *V, int64_t batch, int64_t seq,
                         int64_t heads, int64_t dim, double scale, int causal, const int64_t *rows,
                         int64_t n_rows, double *out, double *bound, int nthreads) {
  if (batch < 0 || seq < 0 || heads < 0 || dim < 0 || n_rows < 0) return -1;
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t i = rows ? rows[r] : r;
    if (i < 0 || i >= seq) return -1;
  }
  const int64_t items = batch * n_rows * heads;
  if (items == 0 || dim == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > items) nthreads = (int)items;

  oracle_attn_job *jobs = (oracle_attn_job *)calloc((size_t)nthreads, sizeof(oracle_attn_job));
  pthread_t *threads = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !threads) {
    free(jobs);
    free(threads);
    return -1;
  }
  int status = 0;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    oracle_attn_job *j = &jobs[t];
    j->Q = Q;
    j->K = K;
    j->V = V;
    j->batch = batch;
    j->seq = seq;
    j->heads = heads;
    j->dim = dim;
    j->scale = scale;
    j->causal = causal;
    j->rows = rows;
    j->n_rows = n_rows;
    j->out = out;
    j->bound = bound;
    j->item_begin = items * t / nthreads;
    j->item_end = items * (t + 1) / nthreads;
    if (t == 0) continue; /* the calling thread takes the first slice */
    if (pthread_create(&threads[t], NULL, oracle_attn_thread, j) != 0) {
      status = -1;
      break;
    }
    started = t;
  }
  if (status == 0) oracle_attn_items(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(threads[t], NULL);
  for (int t = 0; t <= started; ++t)
    if (jobs[t].status != 0) status = -1;
  free(jobs);
  free(threads);
  return status;
}
