// sm103_gemm_fused.cu -- instantiations of the tcgen05 GEMM kernel with the
// fused epilogue D = act(alpha * A x B^T + beta * C + bias[j]) (the pair
// 256 x 256 and single-CTA 128 x 128 configurations), and the elementwise
// kernel that gives the same epilogue its meaning when K = 0.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_tn_internal.h"
#include "sm103_launch.cuh"

namespace gemm_tn_dev {

// K = 0: the product is the empty sum, so D = act(beta * C + bias[j]).
template <typename T>
__global__ void __launch_bounds__(256) fused_k0_kernel(T* c, int64_t ldc, float* c32, int64_t m, int64_t n, float beta,
                                                       const float* bias, int activation) {
  const int64_t total = m * n;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = idx / n, j = idx - (idx / n) * n;
    const int64_t at = i * ldc + j;
    float v = bias != nullptr ? bias[j] : 0.0f;
    if (beta != 0.0f) v += beta * (c32 != nullptr ? c32[at] : static_cast<float>(c[at]));
    if (activation == 1) v = fmaxf(v, 0.0f);
    if (activation == 2) v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
    if (c32 != nullptr) {
      c32[at] = v;
    } else {
      c[at] = static_cast<T>(v);
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

cudaError_t launch_fused_k0(bool bf16, void* c, int64_t ldc, bool out_f32, int64_t m, int64_t n, float beta,
                            const float* bias, int activation, int num_sms, cudaStream_t stream) {
  const int64_t total = m * n;
  const int64_t max_grid = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 4;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>((total + 255) / 256, max_grid));
  float* c32 = out_f32 ? static_cast<float*>(c) : nullptr;
  if (bf16) {
    gemm_tn_dev::fused_k0_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<__nv_bfloat16*>(c), ldc, c32, m,
                                                                          n, beta, bias, activation);
  } else {
    gemm_tn_dev::fused_k0_kernel<__half><<<grid, 256, 0, stream>>>(static_cast<__half*>(c), ldc, c32, m, n, beta, bias,
                                                                   activation);
  }
  return cudaGetLastError();
}

}  // namespace gemm_tn_impl
