// repack.cu -- stream-ordered row repack for operands whose layout the
// tensor-memory-access engine cannot describe (base not 16-byte aligned, or a
// row pitch that is not a multiple of 16 bytes). Each row of `cols` 16-bit
// elements is copied to a destination whose pitch `ld_dst` is a multiple of 8
// elements; the padding columns are written as zeros. HBM-bound: every source
// element is read once and every destination element written once.
//
// "Tiling a matmul", section "Where it breaks" (edge tiles need padding or
// predicated loads): this is the padding half, used only for misaligned
// operands; ragged tile edges are handled by the GEMM kernel's bounded loads.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_tn_internal.h"

namespace gemm_tn_dev {

// One CTA walks whole rows; consecutive threads take consecutive 16-byte
// chunks of a destination row, so the stores are full 16-byte vectors and the
// 2-byte loads of a warp cover one contiguous 512-byte span of the source row.
__global__ void __launch_bounds__(256) repack_rows_kernel(const uint16_t* __restrict__ src, int64_t ld_src,
                                                          uint16_t* __restrict__ dst, int64_t ld_dst, int64_t rows,
                                                          int64_t cols) {
  const int64_t chunks = ld_dst / 8;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint16_t* s = src + r * ld_src;
    uint4* d = reinterpret_cast<uint4*>(dst + r * ld_dst);
    for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) {
      const int64_t c0 = c * 8;
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t e0 = c0 + 2 * j, e1 = e0 + 1;
        const uint32_t lo = e0 < cols ? s[e0] : 0u;
        const uint32_t hi = e1 < cols ? s[e1] : 0u;
        w[j] = lo | (hi << 16);
      }
      d[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace gemm_tn_dev

namespace gemm_tn_impl {

cudaError_t launch_repack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows, int64_t cols,
                          int num_sms, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int64_t max_grid = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
  const unsigned grid = static_cast<unsigned>(rows < max_grid ? rows : max_grid);
  gemm_tn_dev::repack_rows_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(src), ld_src,
                                                             static_cast<uint16_t*>(dst), ld_dst, rows, cols);
  return cudaGetLastError();
}

}  // namespace gemm_tn_impl
