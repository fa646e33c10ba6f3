// sm103_gemm_1cta.cu -- instantiations of the tcgen05 GEMM kernel with one CTA
// per output tile (cta_group::1): 128 x 256, 128 x 128 and 128 x 64 tiles, the
// last two also with two k-blocks per stage.
#include "gemm_tn_internal.h"
#include "sm103_launch.cuh"

namespace gemm_tn_impl {

using Cfg256F16 = gemm_tn_dev::GemmConfig<1, 256, 4, false>;
using Cfg256Bf16 = gemm_tn_dev::GemmConfig<1, 256, 4, true>;
using Cfg128F16 = gemm_tn_dev::GemmConfig<1, 128, 6, false>;
using Cfg128Bf16 = gemm_tn_dev::GemmConfig<1, 128, 6, true>;
using Cfg64F16 = gemm_tn_dev::GemmConfig<1, 64, 8, false>;
using Cfg64Bf16 = gemm_tn_dev::GemmConfig<1, 64, 8, true>;
// two k-blocks per stage: half the stages in the same shared memory (128 x
// 128 and 128 x 64 tiles; 128 x 256 tiles would keep only two stages, and
// ran 18% slower so at 2048^3)
template <int kBlockN, int kStages, bool kBf16>
using CfgPairs = gemm_tn_dev::GemmConfig<1, kBlockN, kStages, kBf16, 1, false, false, false, true>;

cudaError_t launch_gemm_1cta(int id, bool bf16, bool k_pairs, const gemm_tn_dev::GemmArgs& args, int grid,
                             cudaStream_t stream) {
  if (k_pairs) {
    switch (id) {
      case kCfg1CtaN128:
        return bf16 ? Launcher<CfgPairs<128, 3, true>>::launch(args, grid, stream)
                    : Launcher<CfgPairs<128, 3, false>>::launch(args, grid, stream);
      case kCfg1CtaN64:
        return bf16 ? Launcher<CfgPairs<64, 4, true>>::launch(args, grid, stream)
                    : Launcher<CfgPairs<64, 4, false>>::launch(args, grid, stream);
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (id) {
    case kCfg1CtaN256:
      return bf16 ? Launcher<Cfg256Bf16>::launch(args, grid, stream) : Launcher<Cfg256F16>::launch(args, grid, stream);
    case kCfg1CtaN128:
      return bf16 ? Launcher<Cfg128Bf16>::launch(args, grid, stream) : Launcher<Cfg128F16>::launch(args, grid, stream);
    case kCfg1CtaN64:
      return bf16 ? Launcher<Cfg64Bf16>::launch(args, grid, stream) : Launcher<Cfg64F16>::launch(args, grid, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

static_assert(CfgPairs<128, 3, false>::kSmemBytes <= Cfg128F16::kSmemBytes &&
                  CfgPairs<64, 4, false>::kSmemBytes <= Cfg64F16::kSmemBytes,
              "the paired stages take no more shared memory (occupancy queries use the single form)");

int max_resident_1cta(int id, bool bf16) {
  switch (id) {
    case kCfg1CtaN256:
      return bf16 ? Launcher<Cfg256Bf16>::max_clusters() : Launcher<Cfg256F16>::max_clusters();
    case kCfg1CtaN128:
      return bf16 ? Launcher<Cfg128Bf16>::max_clusters() : Launcher<Cfg128F16>::max_clusters();
    case kCfg1CtaN64:
      return bf16 ? Launcher<Cfg64Bf16>::max_clusters() : Launcher<Cfg64F16>::max_clusters();
    default:
      return 0;
  }
}

int smem_bytes_1cta(int id) {
  return id == kCfg1CtaN256  ? static_cast<int>(Cfg256F16::kSmemBytes)
         : id == kCfg1CtaN64 ? static_cast<int>(Cfg64F16::kSmemBytes)
                              : static_cast<int>(Cfg128F16::kSmemBytes);
}

}  // namespace gemm_tn_impl
