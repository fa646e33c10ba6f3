/*
 * flash_attn.h -- C ABI of the attention forward pass that runs on the
 * gemm_tn pipeline (same library, libgemm_tn.so, and the same status codes).
 *
 * Operation ("TileLang: a tile language one level below Triton", section
 * "FlashAttention: online softmax as tile code"): for every batch b < B, head
 * h < H and query position i < S,
 *
 *     s_j            = scale * sum_d Q[b][i][h][d] * K[b][j][h][d]   (visible j)
 *     O[b][i][h][d]  = sum_j softmax(s)_j * V[b][j][h][d]
 *
 * where the visible keys are j <= i when `causal` is non-zero (the section's
 * mask: a score is kept when the query index is at least the key index) and
 * every j < S otherwise. Q, K, V and O are [B, S, H, D] arrays (D = head_dim
 * contiguous, then heads, then positions, then batches), fp16 or bf16.
 * Scores, the softmax's running maximum and row sum, and the output
 * accumulator are fp32; the probabilities are rounded to the input type before
 * the product with V (the section's fp16 probabilities), and O is rounded to
 * nearest-even into the input type. Against the exact result every element
 * satisfies |o - ref| <= 1e-2 * sum_j p_j * |V[b][j][h][d]| + 1e-3.
 *
 * Conventions (as in gemm_tn.h):
 *   - Device pointers are caller-owned; nothing is retained after a call.
 *     Q, K, V and O must be 16-byte aligned; O must not overlap Q, K or V.
 *   - The work is enqueued on `stream` and the call returns without waiting.
 *   - B, S or H equal to 0 does nothing and returns GEMM_TN_OK.
 *   - Host-side errors are the return value and nothing is enqueued:
 *       GEMM_TN_ERR_INVALID_VALUE   negative size, head_dim not 64 or 128, a
 *                                   NULL pointer, O overlapping an input,
 *                                   softmax_scale negative or not finite, or
 *                                   sizes past the limits (S < 2^31,
 *                                   B * H * ceil(S / 128) < 2^31, one
 *                                   [S, H, D] batch under 2^39 bytes);
 *       GEMM_TN_ERR_UNSUPPORTED_DTYPE, GEMM_TN_ERR_MISALIGNED,
 *       GEMM_TN_ERR_UNSUPPORTED_DEVICE, GEMM_TN_ERR_CUDA.
 *   - The device watchdog bounds every wait (GEMM_TN_WATCHDOG_MS, default
 *     4 s); when one expires the kernel stops, O is unspecified, and
 *     GEMM_TN_ERR_TIMEOUT is stored in *d_status if d_status is not NULL.
 *     GEMM_TN_TEST_DROP_LOAD=<tile> is a test hook: the first CTA skips the K
 *     load of that key tile so that a wait expires.
 *   - Only compute capability 10.3 (GB300) devices are supported.
 */
#ifndef FLASH_ATTN_H_
#define FLASH_ATTN_H_

#include <stdint.h>

#include "gemm_tn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * flash_attn_fwd -- O = softmax(scale * Q K^T, mask) V, per batch and head.
 * dtype: GEMM_TN_F16 or GEMM_TN_BF16 (Q, K, V and O alike).
 * batch, seq, heads, head_dim: B, S, H, D (D = 64 or 128).
 * q, k, v: device [B, S, H, D] inputs; o: device [B, S, H, D] output.
 * softmax_scale: the factor on Q.K; 0 selects 1/sqrt(head_dim).
 * causal: non-zero applies the causal mask (query i sees keys j <= i).
 * d_status: optional device int for the watchdog (may be NULL).
 */
GEMM_TN_API int flash_attn_fwd(int dtype, int64_t batch, int64_t seq, int64_t heads, int64_t head_dim, const void* q,
                               const void* k, const void* v, void* o, float softmax_scale, int causal, int* d_status,
                               gemm_tn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FLASH_ATTN_H_ */
