// sm103_gemm_2cta.cu -- instantiations of the tcgen05 GEMM kernel with a CTA
// pair (cta_group::2, two SMs) per 256 x 256 or 256 x 128 output tile, and the
// 4-CTA cluster variant whose two pairs share A through TMA multicast.
#include "gemm_tn_internal.h"
#include "sm103_launch.cuh"

namespace gemm_tn_impl {

using CfgPairF16 = gemm_tn_dev::GemmConfig<2, 256, 6, false>;
using CfgPairBf16 = gemm_tn_dev::GemmConfig<2, 256, 6, true>;
using CfgPair128F16 = gemm_tn_dev::GemmConfig<2, 128, 8, false>;
using CfgPair128Bf16 = gemm_tn_dev::GemmConfig<2, 128, 8, true>;
// two pairs per cluster sharing A through TMA multicast
using CfgPairMcF16 = gemm_tn_dev::GemmConfig<2, 256, 6, false, 2>;
using CfgPairMcBf16 = gemm_tn_dev::GemmConfig<2, 256, 6, true, 2>;
// the same two configurations able to run the cut sub-tiles of a last wave
using CfgPairSplitF16 = gemm_tn_dev::GemmConfig<2, 256, 6, false, 1, false, false, true>;
using CfgPairSplitBf16 = gemm_tn_dev::GemmConfig<2, 256, 6, true, 1, false, false, true>;
using CfgPairMcSplitF16 = gemm_tn_dev::GemmConfig<2, 256, 6, false, 2, false, false, true>;
using CfgPairMcSplitBf16 = gemm_tn_dev::GemmConfig<2, 256, 6, true, 2, false, false, true>;

cudaError_t launch_gemm_2cta(int id, bool bf16, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
  if (args.split > 1) {
    switch (id) {
      case kCfg2CtaN256:
        return bf16 ? Launcher<CfgPairSplitBf16>::launch(args, grid, stream)
                    : Launcher<CfgPairSplitF16>::launch(args, grid, stream);
      case kCfg2CtaN256Mc:
        return bf16 ? Launcher<CfgPairMcSplitBf16>::launch(args, grid, stream)
                    : Launcher<CfgPairMcSplitF16>::launch(args, grid, stream);
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (id) {
    case kCfg2CtaN256:
      return bf16 ? Launcher<CfgPairBf16>::launch(args, grid, stream) : Launcher<CfgPairF16>::launch(args, grid, stream);
    case kCfg2CtaN128:
      return bf16 ? Launcher<CfgPair128Bf16>::launch(args, grid, stream)
                  : Launcher<CfgPair128F16>::launch(args, grid, stream);
    case kCfg2CtaN256Mc:
      return bf16 ? Launcher<CfgPairMcBf16>::launch(args, grid, stream)
                  : Launcher<CfgPairMcF16>::launch(args, grid, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

int max_resident_2cta(int id, bool bf16) {
  switch (id) {
    case kCfg2CtaN256:
      return bf16 ? Launcher<CfgPairBf16>::max_clusters() : Launcher<CfgPairF16>::max_clusters();
    case kCfg2CtaN128:
      return bf16 ? Launcher<CfgPair128Bf16>::max_clusters() : Launcher<CfgPair128F16>::max_clusters();
    case kCfg2CtaN256Mc:
      return bf16 ? Launcher<CfgPairMcBf16>::max_clusters() : Launcher<CfgPairMcF16>::max_clusters();
    default:
      return 0;
  }
}

int smem_bytes_2cta(int id) {
  return id == kCfg2CtaN256 ? static_cast<int>(CfgPairF16::kSmemBytes) : static_cast<int>(CfgPair128F16::kSmemBytes);
}

}  // namespace gemm_tn_impl
