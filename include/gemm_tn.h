/*
 * gemm_tn.h -- C ABI of a GB300-native (sm_103a) tiled dense GEMM.
 *
 * Operation ("0. A Minimal Hopper Matmul", section "Block Tiling", and its note
 * on K-major data layout):
 *
 *     C[i][j] = sum_{k} A[i][k] * B[j][k]          i < M, j < N, k < K
 *
 * i.e. C = A x B^T with A of shape [M, K] and B of shape [N, K], both K-major
 * (each row contiguous, K elements long, rows `lda` / `ldb` elements apart),
 * and C of shape [M, N] row-major with rows `ldc` elements apart. A and B are
 * fp16 or bf16; products are accumulated in fp32 ("0. A Minimal Hopper
 * Matmul", section "Kernel Setup": fp32 accumulator) and the result is rounded
 * to nearest-even into the input dtype ("Epilogue": cast back to 16 bits).
 * Tiling changes only the order of the additions ("Tiling a matmul", section
 * "Where it breaks"), so results match the exact product within
 * |c - ref| <= 1e-2 * sum_k |a_ik * b_jk| + 1e-3 but are not bit-identical to
 * any particular summation order.
 *
 * Conventions shared by every entry point:
 *   - Sizes are element counts. M, N and K must each be below 2^31.
 *   - Device pointers are caller-owned; nothing is retained after a call.
 *     A, B and C must each be 2-byte aligned. C must not overlap A or B.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Device
 *     work is enqueued on it and the call returns without waiting, except
 *     gemm_tn_host, which waits for its stream.
 *   - M == 0 or N == 0 does nothing and returns GEMM_TN_OK. K == 0 writes
 *     zeros to C (the empty sum).
 *   - Host-side errors are the return value; nothing is enqueued on error.
 *   - Device-side watchdog: every wait inside the kernel is bounded (default
 *     4 s, environment variable GEMM_TN_WATCHDOG_MS). When one expires the
 *     kernel stops, leaves C unspecified and, if the caller passed `d_status`,
 *     stores GEMM_TN_ERR_TIMEOUT there (first error wins; the caller zeroes
 *     it and reads it after synchronising).
 *   - Stream-K tail: when the output tiles fill at least one wave of the
 *     persistent grid and leave a partial last wave, that wave's tiles are
 *     cut into k-block ranges over the workers ("Tiling a matmul", section
 *     "Where it breaks": split-K / stream-K keep all SMs busy); the fp32
 *     partial rows go through a stream-ordered workspace (see
 *     gemm_tn_workspace_pool) and are added in a fixed order, so repeated
 *     calls stay bit-identical.
 *     GEMM_TN_STREAMK=0 turns it off (the last wave's tiles are then cut
 *     along N instead when that fits one wave); 1, 2 or 3 force a mode
 *     (measurements and tests).
 *     The environment variable GEMM_TN_TEST_DROP_LOAD=<k-block> is a test
 *     hook of gemm_tn_ex: the kernel skips that k-block's loads of its first
 *     tiles so that a wait expires and the watchdog path runs.
 *   - Kernels are launched as programmatic dependents of the previous kernel
 *     in `stream`: their set-up may overlap its end, but they touch memory
 *     only once it has completed, so stream order holds as for any launch
 *     (GEMM_TN_PDL=0 launches them plainly).
 *   - The kernel configuration is chosen per call (gemm_tn_select_config;
 *     gemm_tn_select_splits gives the K split of the split-K ones).
 *     Problems with few output tiles split K over a thread-block cluster and
 *     add the fp32 partials in a fixed order; problems with one row of tiles
 *     start each tile's K walk at a hashed k-block. Each configuration gives
 *     bit-identical results on repeated calls.
 *   - Thread-safe: the shared state is a per-device cache of attributes and
 *     the launch counter (atomic).
 *   - Only compute capability 10.3 (GB300) devices are supported.
 */
#ifndef GEMM_TN_H_
#define GEMM_TN_H_

#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_TN_API __attribute__((visibility("default")))
#else
#define GEMM_TN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* gemm_tn_stream_t;

/* Element type of A, B and C. */
enum gemm_tn_dtype { GEMM_TN_F16 = 0, GEMM_TN_BF16 = 1 };

/* Return / device status codes. */
enum gemm_tn_status {
  GEMM_TN_OK = 0,
  GEMM_TN_ERR_INVALID_VALUE = 1,      /* negative or too-large size, NULL pointer with non-zero size,
                                         leading dimension too small, C overlapping A or B */
  GEMM_TN_ERR_UNSUPPORTED_DTYPE = 2,  /* dtype is neither GEMM_TN_F16 nor GEMM_TN_BF16 */
  GEMM_TN_ERR_MISALIGNED = 3,         /* a pointer is not 2-byte aligned */
  GEMM_TN_ERR_UNSUPPORTED_DEVICE = 4, /* no current device, or it is not compute capability 10.3 */
  GEMM_TN_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed: see gemm_tn_last_cuda_error() */
  GEMM_TN_ERR_TIMEOUT = 6             /* device watchdog expired (written to *d_status only) */
};

/*
 * gemm_tn -- C = A x B^T for contiguous operands: lda = ldb = k, ldc = n.
 * a: device [m, k]; b: device [n, k]; c: device [m, n] (written).
 */
GEMM_TN_API int gemm_tn(int dtype, int64_t m, int64_t n, int64_t k, const void* a, const void* b, void* c,
            gemm_tn_stream_t stream);

/*
 * gemm_tn_ex -- C = A x B^T with explicit row strides (in elements):
 * lda >= k, ldb >= k, ldc >= n. Any stride and any 2-byte-aligned pointer is
 * accepted. When A or B is not laid out the way the tensor-memory-access
 * engine needs (16-byte-aligned base, row pitch a multiple of 16 bytes) the
 * call first copies that operand into a stream-ordered workspace with a
 * padded row pitch (allocated and freed on `stream` in the library's
 * workspace pool, gemm_tn_workspace_pool).
 * d_status: nullable device int that receives GEMM_TN_ERR_TIMEOUT if the
 * device watchdog fires; never cleared by the library.
 */
GEMM_TN_API int gemm_tn_ex(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda, const void* b,
               int64_t ldb, void* c, int64_t ldc, int* d_status, gemm_tn_stream_t stream);

/* Fused epilogue of gemm_tn_fused. */
enum gemm_tn_activation { GEMM_TN_ACT_NONE = 0, GEMM_TN_ACT_RELU = 1, GEMM_TN_ACT_GELU = 2 };
enum gemm_tn_out_dtype { GEMM_TN_OUT_INPUT = 0, GEMM_TN_OUT_F32 = 1, GEMM_TN_OUT_E4M3 = 2 };
typedef struct gemm_tn_epilogue {
  float alpha;        /* scale of A x B^T */
  float beta;         /* scale of C's previous contents; 0: C is not read */
  const float* bias;  /* nullable device fp32 [n], added to every row */
  int activation;     /* GEMM_TN_ACT_*: none, max(x, 0), or x * Phi(x) (erf form) */
  int out_dtype;      /* GEMM_TN_OUT_INPUT: C has A's dtype; GEMM_TN_OUT_F32: C is fp32;
                         GEMM_TN_OUT_E4M3: C is fp8 e4m3 (1 sign, 4 exponent bits with bias 7,
                         3 mantissa bits; largest finite 448, no infinities) */
} gemm_tn_epilogue;

/*
 * gemm_tn_fused -- D = act(alpha * (A x B^T) + beta * C + bias[j]) written
 * over C, all in fp32 in the GEMM's epilogue before the one rounding to C's
 * dtype: the step after the GEMM done without another pass over C. A and B
 * as in gemm_tn_ex; C has ldc >= n elements per row of out_dtype and is
 * aligned to that element (4 bytes for fp32, 2 for fp16/bf16, none for e4m3).
 * The e4m3 output is the fused form of a quantising pass after the GEMM:
 * alpha carries the caller's quantisation scale, D rounds to nearest even
 * with saturation (|D| past 448 stores +-448, NaN stays NaN), and with
 * beta != 0 C's previous e4m3 contents are read back exactly. ("TileLang: a
 * tile language one level below Triton", exercise 4: a quantisation to FP8
 * is bandwidth-bound, so it belongs fused with the operator that produces
 * its input.) K == 0 gives act(beta * C + bias). Same errors, watchdog,
 * workspace and stream-K behaviour as gemm_tn_ex (with a stream-K tail the
 * fp32 partial sums are added before the epilogue's one pass over C).
 */
GEMM_TN_API int gemm_tn_fused(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda, const void* b,
                              int64_t ldb, void* c, int64_t ldc, const gemm_tn_epilogue* epilogue, int* d_status,
                              gemm_tn_stream_t stream);

/*
 * gemm_nn -- C = A x B with B stored [K, N], N contiguous (rows ldb >= n
 * elements apart): C[i][j] = sum_k A[i][k] * B[k][j]. A and C as in
 * gemm_tn_ex. The kernel reads B in that layout directly (MN-major operand
 * descriptors), with no transpose pass; the GEMM the TileLang page writes
 * ("TileLang: a tile language one level below Triton", section "The first
 * kernel: GEMM", B declared (K, N)). Arguments, errors, watchdog and
 * workspace behaviour are those of gemm_tn_ex.
 */
GEMM_TN_API int gemm_nn(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda, const void* b,
                        int64_t ldb, void* c, int64_t ldc, int* d_status, gemm_tn_stream_t stream);

/*
 * gemm_tn_ex_noalloc -- gemm_tn_ex for callers that cannot allocate device
 * memory: the pages this library follows have no counterpart of it.
 *
 * Some callers must not call cudaMalloc or cudaMallocAsync: a framework that
 * has reserved (nearly) all device memory for its own pool at start-up, where
 * an extra allocation fails or fragments the pool, or a code path with a hard
 * latency or memory budget, where an allocation can block or fail at the
 * worst moment. This entry point computes the product gemm_tn_ex computes,
 * with the same arguments and checks, and allocates nothing: the padded copy
 * of an operand whose base or row pitch the tensor-memory-access engine
 * cannot address comes from a static device array of
 * GEMM_TN_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU loading this library
 * holds until the process exits, and the stream-K tail (which needs a
 * workspace) is not used: a partial last wave of tiles is cut along N or run
 * whole instead, so the low-order bits of those tiles can differ from
 * gemm_tn_ex's (both are within the stated tolerance).
 *
 * - The first call on a device looks up that array's device address (with
 *   the device current) and caches it with the current context; make that
 *   first call before any stream capture on the device. A call under another
 *   context of the device (one the caller created, or the primary context
 *   again after cudaDeviceReset) repeats the lookup for that context.
 * - A problem whose repacked operands need more than
 *   GEMM_TN_NOALLOC_SCRATCH_BYTES is rejected with GEMM_TN_ERR_INVALID_VALUE
 *   and nothing is enqueued. Operands that need no repack use no scratch.
 * - All calls share the one array and it keeps the last call's contents
 *   (every byte a call reads is written by that call first). Calls whose GPU
 *   work overlaps in time (different streams, or threads) race on it:
 *   serialise them, e.g. on one stream.
 */
#define GEMM_TN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
GEMM_TN_API int gemm_tn_ex_noalloc(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda,
                                   const void* b, int64_t ldb, void* c, int64_t ldc, int* d_status,
                                   gemm_tn_stream_t stream);

/*
 * gemm_tn_host -- C = A x B^T with contiguous operands in HOST memory
 * (pinned for full copy speed; pageable works): copies A and B to the current
 * device, computes, copies C back and waits for everything before returning.
 * B is copied first, then A in chunks of rows; each chunk's GEMM runs on
 * `stream` while the next chunk of A is copied in and the previous chunk of C
 * is copied out on two library-owned copy streams. Device staging memory comes
 * from a library-owned pool that keeps it for later calls. Calls on one device
 * are serialised. Returns GEMM_TN_ERR_TIMEOUT if the watchdog fired.
 */
GEMM_TN_API int gemm_tn_host(int dtype, int64_t m, int64_t n, int64_t k, const void* a_host, const void* b_host,
                 void* c_host, gemm_tn_stream_t stream);

/* Kernel configuration gemm_tn_ex would run for this problem on the current
 * device (an index into the table below), or -1 for a no-op / invalid size.
 * The environment variable GEMM_TN_FORCE_CONFIG (a name or an index)
 * overrides the table. */
GEMM_TN_API int gemm_tn_select_config(int dtype, int64_t m, int64_t n, int64_t k);

/* K split gemm_tn_ex would run for this problem on the current device when
 * the chosen configuration is a split-K one (1cta_n128_splitk or
 * 1cta_decode_splitk): the number of CTAs of a cluster that share one
 * output tile's K (2, 4 or 8). 0 for every other configuration, or for a
 * no-op / invalid size. GEMM_TN_FORCE_CONFIG and GEMM_TN_SPLITK apply as in
 * gemm_tn_ex. Host-only: launches nothing. */
GEMM_TN_API int gemm_tn_select_splits(int dtype, int64_t m, int64_t n, int64_t k);

/* The memory pool (a cudaMemPool_t, returned as void*) that the calls above
 * take their stream-ordered workspaces from on the current device: padded
 * copies of misaligned operands and the stream-K tail's fp32 partials. The
 * library creates it on first use (pinned device memory of that device) and
 * never returns its memory on its own: a workspace freed by one call is reused
 * by the next without mapping memory again. Its attributes can be read with
 * cudaMemPoolGetAttribute (diagnostics). NULL when there is no usable device. */
GEMM_TN_API void* gemm_tn_workspace_pool(void);

/* Return the workspace pool's unused memory on the current device to the
 * system (cudaMemPoolTrimTo(pool, 0)); memory of workspaces still in use on
 * some stream is kept. GEMM_TN_ERR_CUDA / _UNSUPPORTED_DEVICE on failure. */
GEMM_TN_API int gemm_tn_trim_workspace(void);

/* Kernel configuration (an index into the table below) that the calling
 * thread's last gemm_tn / gemm_tn_ex / gemm_tn_fused / gemm_nn /
 * gemm_tn_ex_noalloc call launched, or -1 if that call launched no GEMM kernel
 * (an error, an empty problem or K == 0). gemm_tn_host reports the
 * configuration of its last row chunk. Diagnostics; never fails. */
GEMM_TN_API int gemm_tn_last_config(void);

/*
 * Whether the multicast configuration ("2cta_n256_mc") may read A and B: 1
 * when both are device memory of the current device, else 0 (host or managed
 * memory, another GPU's memory reached through peer access, an unknown
 * pointer, or no usable device). In that configuration one CTA loads a
 * half-tile of A for two CTA pairs with a cluster-multicast TMA load ("Tiling a
 * matmul", section "The levels of tiling": a cluster shares a tile between its
 * CTAs); such loads are issued only on this GPU's own memory. Every GEMM entry
 * point applies this check whenever the selection (or GEMM_TN_FORCE_CONFIG)
 * picks that configuration, and runs the plain CTA-pair configuration
 * ("2cta_n256") when it fails. Host-only: launches nothing.
 */
GEMM_TN_API int gemm_tn_multicast_allowed(const void* a, const void* b);

/* Number of kernel configurations, and the name of one ("1cta_n256", ...,
 * "1cta_n128_splitk": K split over a cluster of 2, 4 or 8 CTAs per 128 x 128
 * tile, chosen when the tiles fill less than half the SMs; "1cta_decode_splitk":
 * the same split with B's rows on the MMA's M side, for M <= 32; "1cta_n64":
 * 128 x 64 tiles for problems whose tiles fill at most half the SMs). */
GEMM_TN_API int gemm_tn_num_configs(void);
GEMM_TN_API const char* gemm_tn_config_name(int config);

/* Human-readable text of a status code. */
GEMM_TN_API const char* gemm_tn_status_string(int status);

/* cudaError_t of the last failing CUDA call made by this thread (0 if none),
 * and a one-line description of the last error this thread returned. */
GEMM_TN_API int gemm_tn_last_cuda_error(void);
GEMM_TN_API const char* gemm_tn_last_error_message(void);

/* ABI version: major * 100 + minor. */
GEMM_TN_API int gemm_tn_version(void);

/* Number of kernels this library has launched in this process so far, over
 * every thread and device: GEMM kernels (one per call), repack
 * kernels for misaligned operands, the K = 0 epilogue kernel and attention
 * kernels. Diagnostics: read it before and after a region of work to count
 * that region's launches. Never fails. */
GEMM_TN_API uint64_t gemm_tn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_TN_H_ */
