// sm103_gemm_2cta.cu -- instantiations of the tcgen05 GEMM kernel with a CTA
// pair (a 2-CTA cluster on two SMs, cta_group::2) per 256 x 256 output tile.
#include "gemm_tn_internal.h"
#include "sm103_launch.cuh"

namespace gemm_tn_impl {

using CfgPairF16 = gemm_tn_dev::GemmConfig<2, 256, 6, false>;
using CfgPairBf16 = gemm_tn_dev::GemmConfig<2, 256, 6, true>;

cudaError_t launch_gemm_2cta(int id, bool bf16, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
  if (id != kCfg2CtaN256) return cudaErrorInvalidValue;
  return bf16 ? Launcher<CfgPairBf16>::launch(args, grid, stream) : Launcher<CfgPairF16>::launch(args, grid, stream);
}

int max_resident_2cta(int id, bool bf16) {
  if (id != kCfg2CtaN256) return 0;
  return bf16 ? Launcher<CfgPairBf16>::max_clusters() : Launcher<CfgPairF16>::max_clusters();
}

int smem_bytes_2cta(int /*id*/) { return static_cast<int>(CfgPairF16::kSmemBytes); }

}  // namespace gemm_tn_impl
