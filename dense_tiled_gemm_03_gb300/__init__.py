"""GB300-native tiled dense GEMM, C = A x B^T (A [M,K], B [N,K], K-major,
fp16/bf16 in, fp32 accumulate, fp16/bf16 out), and the attention forward pass
built on the same pipeline (``flash_attn``).

The product is the C-ABI library ``libgemm_tn.so`` (hand-written sm_103a CUDA:
TMA, mbarrier rings, tcgen05 tensor cores with TMEM accumulators); this
package is its ctypes binding plus the seeded workload generator. Build the
library with ``python -m dense_tiled_gemm_03_gb300.build``.
"""
from ._native import (  # noqa: F401
    GEMM_TN_BF16,
    GEMM_TN_ERR_CUDA,
    GEMM_TN_ERR_INVALID_VALUE,
    GEMM_TN_ERR_MISALIGNED,
    GEMM_TN_ERR_TIMEOUT,
    GEMM_TN_ERR_UNSUPPORTED_DEVICE,
    GEMM_TN_ERR_UNSUPPORTED_DTYPE,
    GEMM_TN_F16,
    GEMM_TN_OK,
    GEMM_TN_OUT_E4M3,
    GEMM_TN_OUT_F32,
    GEMM_TN_OUT_INPUT,
    LIBRARY_PATH,
    GemmTnEpilogue,
    GemmTnError,
    flash_attn,
    flash_attn_fwd,
    gemm_nn,
    gemm_tn_fused,
    gemm_tn,
    gemm_tn_config_name,
    gemm_tn_ex,
    gemm_tn_ex_noalloc,
    GEMM_TN_NOALLOC_SCRATCH_BYTES,
    gemm_tn_host,
    gemm_tn_last_cuda_error,
    gemm_tn_last_config,
    gemm_tn_last_error_message,
    gemm_tn_multicast_allowed,
    gemm_tn_trim_workspace,
    gemm_tn_workspace_pool,
    gemm_tn_num_configs,
    gemm_tn_select_config,
    gemm_tn_select_splits,
    gemm_tn_status_string,
    gemm_tn_version,
    gemm_tn_launch_count,
    library,
    mm_nn,
    mm_tn_fused,
    mm_tn,
    mm_tn_host,
)
