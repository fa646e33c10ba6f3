// sm103_gemm_fused.cu -- instantiations of the tcgen05 GEMM kernel with the
// fused epilogue D = act(alpha * A x B^T + beta * C + bias[j]), stored as the
// input dtype, fp32 or saturating fp8 e4m3 (the pair
// 256 x 256 and single-CTA 128 x 128 configurations), and the elementwise
// kernel that gives the same epilogue its meaning when K = 0.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_tn_internal.h"
#include "sm103_launch.cuh"

namespace gemm_tn_dev {

// K = 0: the product is the empty sum, so D = act(beta * C + bias[j]), with C
// of element type out_kind (0 T, 1 fp32, 2 e4m3).
template <typename T>
__global__ void __launch_bounds__(256) fused_k0_kernel(void* c, int64_t ldc, int out_kind, int64_t m, int64_t n,
                                                       float beta, const float* bias, int activation) {
  const int64_t total = m * n;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = idx / n, j = idx - (idx / n) * n;
    const int64_t at = i * ldc + j;
    float v = bias != nullptr ? bias[j] : 0.0f;
    if (beta != 0.0f) {
      float prev;
      if (out_kind == 1) {
        prev = static_cast<const float*>(c)[at];
      } else if (out_kind == 2) {
        float unused;
        e4m3x2_to_f32(static_cast<const uint8_t*>(c)[at], prev, unused);
      } else {
        prev = static_cast<float>(static_cast<const T*>(c)[at]);
      }
      v += beta * prev;
    }
    if (activation == 1) v = fmaxf(v, 0.0f);
    if (activation == 2) v = gelu_erf(v);
    if (out_kind == 1) {
      static_cast<float*>(c)[at] = v;
    } else if (out_kind == 2) {
      static_cast<uint8_t*>(c)[at] = static_cast<uint8_t>(cvt_e4m3x2(v, 0.0f));
    } else {
      static_cast<T*>(c)[at] = static_cast<T>(v);
    }
  }
}

}  // namespace gemm_tn_dev

namespace gemm_tn_impl {

template <bool kBf16>
using Fused2Cta256 = gemm_tn_dev::GemmConfig<2, 256, 6, kBf16, 1, false, true>;
template <bool kBf16>
using Fused1Cta128 = gemm_tn_dev::GemmConfig<1, 128, 6, kBf16, 1, false, true>;

cudaError_t launch_gemm_fused(int id, bool bf16, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
  switch (id) {
    case kCfg2CtaN256:
      return bf16 ? Launcher<Fused2Cta256<true>>::launch(args, grid, stream)
                  : Launcher<Fused2Cta256<false>>::launch(args, grid, stream);
    case kCfg1CtaN128:
      return bf16 ? Launcher<Fused1Cta128<true>>::launch(args, grid, stream)
                  : Launcher<Fused1Cta128<false>>::launch(args, grid, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fused_k0(bool bf16, void* c, int64_t ldc, int out_kind, int64_t m, int64_t n, float beta,
                            const float* bias, int activation, int num_sms, cudaStream_t stream) {
  const int64_t total = m * n;
  const int64_t max_grid = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 4;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>((total + 255) / 256, max_grid));
  if (bf16) {
    gemm_tn_dev::fused_k0_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(c, ldc, out_kind, m, n, beta, bias,
                                                                          activation);
  } else {
    gemm_tn_dev::fused_k0_kernel<__half><<<grid, 256, 0, stream>>>(c, ldc, out_kind, m, n, beta, bias, activation);
  }
  return cudaGetLastError();
}

}  // namespace gemm_tn_impl
