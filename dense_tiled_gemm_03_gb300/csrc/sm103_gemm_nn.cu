// sm103_gemm_nn.cu -- instantiations of the tcgen05 GEMM kernel with B stored
// [K, N], N contiguous (C = A x B): every configuration of the frozen table,
// with B loaded in 64 x 64 boxes and read through MN-major descriptors.
#include "gemm_tn_internal.h"
#include "sm103_launch.cuh"

namespace gemm_tn_impl {

template <bool kBf16>
using Nn1Cta256 = gemm_tn_dev::GemmConfig<1, 256, 4, kBf16, 1, true>;
template <bool kBf16>
using Nn1Cta128 = gemm_tn_dev::GemmConfig<1, 128, 6, kBf16, 1, true>;
template <bool kBf16>
using Nn2Cta256 = gemm_tn_dev::GemmConfig<2, 256, 6, kBf16, 1, true>;
template <bool kBf16>
using Nn2Cta128 = gemm_tn_dev::GemmConfig<2, 128, 8, kBf16, 1, true>;
template <bool kBf16>
using Nn2Cta256Mc = gemm_tn_dev::GemmConfig<2, 256, 6, kBf16, 2, true>;

template <bool kBf16>
cudaError_t launch_nn(int id, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
  switch (id) {
    case kCfg1CtaN256: return Launcher<Nn1Cta256<kBf16>>::launch(args, grid, stream);
    case kCfg1CtaN128: return Launcher<Nn1Cta128<kBf16>>::launch(args, grid, stream);
    case kCfg2CtaN256: return Launcher<Nn2Cta256<kBf16>>::launch(args, grid, stream);
    case kCfg2CtaN128: return Launcher<Nn2Cta128<kBf16>>::launch(args, grid, stream);
    case kCfg2CtaN256Mc: return Launcher<Nn2Cta256Mc<kBf16>>::launch(args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_nn(int id, bool bf16, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
  return bf16 ? launch_nn<true>(id, args, grid, stream) : launch_nn<false>(id, args, grid, stream);
}

}  // namespace gemm_tn_impl
