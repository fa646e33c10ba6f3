/*
 * gemm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * The plain, slow, obviously correct CPU oracle for the tiled matrix product
 * C = A x B^T with A [M,K] and B [N,K], both K-major (K contiguous in memory).
 * Only tests/, the smoke check and the CPU-baseline leg of the benchmark use it;
 * the product path never links or calls it, and it shares no code with the CUDA
 * library.
 *
 * What it computes (the definition, written out):
 *   "0. A Minimal Hopper Matmul", section "Block Tiling": C = A x B^T with A of
 *   shape (M, K) and B of shape (N, K), output (M, N); section "Data Flow" and
 *   the note on K-major layout: both operands keep K contiguous.
 *   "Tiling a matmul", section "The idea in one minute": tiling only reorders
 *   the same multiply-adds, so the tiled kernel reaches the plain product.
 *
 *     ref[i][j]   = sum_{k=0}^{K-1} A[i][k] * B[j][k]        (fp64, increasing k)
 *     bound[i][j] = sum_{k=0}^{K-1} |A[i][k] * B[j][k]|      (fp64, same loop)
 *
 * The inputs are the fp16/bf16 arrays the GPU sees, widened exactly to fp64 by
 * the caller. Every product of two fp16 (or two bf16) values is exact in fp64,
 * so the only rounding here is the fp64 summation. No blocking, no reordering,
 * no fused multiply-add (built with -ffp-contract=off), no fast-math, no BLAS.
 * Rows are split across plain POSIX threads; each output element is still one
 * sequential dot product, so the thread count never changes a result.
 *
 * ORACLE_PLANT (test builds only, default 0) compiles a deliberate mistake into
 * the loop so the pinning tests can show that each kind of mistake is caught:
 *   1 = drop the last term of every sum, 2 = read B un-transposed (B[k][j]),
 *   3 = subtract the last product instead of adding it, 4 = swap the roles of
 *   i and j in the output index.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

typedef struct {
  const double *A;
  const double *B;
  int64_t M, N, K;
  double *ref;
  double *bound;
  int64_t row_begin, row_end;
} oracle_rows_job;

static void oracle_rows(const oracle_rows_job *job) {
  const int64_t N = job->N, K = job->K;
  for (int64_t i = job->row_begin; i < job->row_end; ++i) {
    const double *a_row = job->A + i * K;
    for (int64_t j = 0; j < N; ++j) {
      double sum = 0.0;
      double abs_sum = 0.0;
      for (int64_t k = 0; k < K; ++k) {
#if ORACLE_PLANT == 1
        if (k == K - 1) break;
#endif
#if ORACLE_PLANT == 2
        /* un-transposed read: only meaningful for square N == K */
        const double b = job->B[k * N + j];
#else
        const double b = job->B[j * K + k];
#endif
        double prod = a_row[k] * b;
#if ORACLE_PLANT == 3
        if (k == K - 1) prod = -prod;
#endif
        sum += prod;
        abs_sum += fabs(prod);
      }
#if ORACLE_PLANT == 4
      const int64_t out = (j < job->M && i < N) ? j * N + i : i * N + j;
#else
      const int64_t out = i * N + j;
#endif
      job->ref[out] = sum;
      job->bound[out] = abs_sum;
    }
  }
}

static void *oracle_rows_thread(void *arg) {
  oracle_rows((const oracle_rows_job *)arg);
  return NULL;
}

/*
 * oracle_gemm_tn_f64: ref[M*N] and bound[M*N] (row-major, leading dim N) from
 * A[M*K] and B[N*K] (row-major, leading dim K), all fp64 host arrays owned by
 * the caller. nthreads <= 0 means one thread. Returns 0, or -1 on bad sizes or
 * a thread that could not be started (then nothing is guaranteed about ref).
 */
int oracle_gemm_tn_f64(const double *A, const double *B, int64_t M, int64_t N,
                       int64_t K, double *ref, double *bound, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (M == 0 || N == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > M) nthreads = (int)M;

  oracle_rows_job *jobs = (oracle_rows_job *)calloc((size_t)nthreads, sizeof(oracle_rows_job));
  pthread_t *threads = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !threads) {
    free(jobs);
    free(threads);
    return -1;
  }
  int status = 0;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].A = A;
    jobs[t].B = B;
    jobs[t].M = M;
    jobs[t].N = N;
    jobs[t].K = K;
    jobs[t].ref = ref;
    jobs[t].bound = bound;
    jobs[t].row_begin = M * t / nthreads;
    jobs[t].row_end = M * (t + 1) / nthreads;
    if (t == 0) continue; /* the calling thread takes the first slice */
    if (pthread_create(&threads[t], NULL, oracle_rows_thread, &jobs[t]) != 0) {
      status = -1;
      break;
    }
    started = t;
  }
  if (status == 0) oracle_rows(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(threads[t], NULL);
  free(jobs);
  free(threads);
  return status;
}
