// repack.cu -- stream-ordered row repack for operands whose layout the
// tensor-memory-access engine cannot describe (base not 16-byte aligned, or a
// row pitch that is not a multiple of 16 bytes). Each row of `cols` 16-bit
// elements is copied to a destination whose pitch `ld_dst` is a multiple of 8
// elements; the padding columns are written as zeros. HBM-bound: every source
// byte is read once from DRAM and every destination byte written once.
//
// "Tiling a matmul", section "Where it breaks" (edge tiles need padding or
// predicated loads): this is the padding half, used only for misaligned
// operands; ragged tile edges are handled by the GEMM kernel's bounded loads.
//
// One launch repacks up to two matrices (A and B). A CTA walks whole rows;
// thread t of the CTA produces 16-byte destination chunks t, t + 256, ... of a
// row. A source row starts at any 2-byte boundary, so each chunk is cut out of
// the two aligned 16-byte source blocks that overlap it (funnel shifts). Only
// aligned blocks holding at least one byte of the row are read, so no access
// leaves the memory the row occupies by more than the rest of its 16-byte block.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_tn_internal.h"

namespace gemm_tn_dev {

struct RepackJob {
  const uint16_t* src;
  int64_t ld_src;
  uint16_t* dst;
  int64_t ld_dst;
  int64_t rows;
  int64_t cols;
};

struct RepackArgs {
  RepackJob job[2];
  int num_jobs;
};

// 16 source bytes, read past L1 and marked first to be evicted from L2: the
// source is read once, so its lines should make room before the copy's
// destination lines, which the GEMM reads right after.
__device__ __forceinline__ uint4 ld_stream(uintptr_t p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// 16 bytes starting `shift` bytes (even, 0..14) into the 32 bytes lo:hi.
__device__ __forceinline__ uint4 extract16(const uint4& lo, const uint4& hi, uint32_t shift) {
  uint32_t x0, x1, x2, x3, x4;
  switch (shift >> 2) {
    case 0: x0 = lo.x; x1 = lo.y; x2 = lo.z; x3 = lo.w; x4 = hi.x; break;
    case 1: x0 = lo.y; x1 = lo.z; x2 = lo.w; x3 = hi.x; x4 = hi.y; break;
    case 2: x0 = lo.z; x1 = lo.w; x2 = hi.x; x3 = hi.y; x4 = hi.z; break;
    default: x0 = lo.w; x1 = hi.x; x2 = hi.y; x3 = hi.z; x4 = hi.w; break;
  }
  const uint32_t bits = (shift & 2u) * 8u;   // 0 or 16
  return make_uint4(__funnelshift_r(x0, x1, bits), __funnelshift_r(x1, x2, bits), __funnelshift_r(x2, x3, bits),
                    __funnelshift_r(x3, x4, bits));
}

__global__ void __launch_bounds__(256) repack_rows_kernel(const __grid_constant__ RepackArgs args) {
  // launched as a programmatic dependent: read the sources only once the
  // previous kernel in the stream has completed; the GEMM that follows may
  // then be scheduled (it waits for this grid before reading the copies)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint64_t evict_first;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
  const int64_t rows_a = args.job[0].rows;
  const int64_t total_rows = rows_a + (args.num_jobs > 1 ? args.job[1].rows : 0);
  for (int64_t gr = blockIdx.x; gr < total_rows; gr += gridDim.x) {
    const RepackJob& jb = args.job[gr < rows_a ? 0 : 1];
    const int64_t r = gr < rows_a ? gr : gr - rows_a;
    const uintptr_t s = reinterpret_cast<uintptr_t>(jb.src + r * jb.ld_src);
    const uintptr_t end = s + static_cast<uintptr_t>(jb.cols) * 2;   // one past the row's last byte
    uint4* d = reinterpret_cast<uint4*>(jb.dst + r * jb.ld_dst);
    const int64_t chunks = jb.ld_dst / 8;
    // two chunks per thread and step, all four source loads issued before
    // either store: the copy is bound by loads in flight (a load's round trip
    // per chunk and thread measured 44% of DRAM bandwidth)
    constexpr int kPer = 2;
    for (int64_t c0 = threadIdx.x; c0 < chunks; c0 += kPer * blockDim.x) {
      uint4 lo[kPer], hi[kPer];
      uint32_t shift[kPer];
      bool inside[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int64_t c = c0 + u * static_cast<int64_t>(blockDim.x);
        const uintptr_t want = s + static_cast<uintptr_t>(c) * 16;
        const uintptr_t base = want & ~static_cast<uintptr_t>(15);
        shift[u] = static_cast<uint32_t>(want - base);
        inside[u] = c < chunks && want < end;
        lo[u] = inside[u] ? ld_stream(base, evict_first) : make_uint4(0u, 0u, 0u, 0u);
        hi[u] = (inside[u] && shift[u] != 0 && base + 16 < end) ? ld_stream(base + 16, evict_first)
                                                                  : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int64_t c = c0 + u * static_cast<int64_t>(blockDim.x);
        if (c >= chunks) continue;
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (inside[u]) {
          out = shift[u] == 0 ? lo[u] : extract16(lo[u], hi[u], shift[u]);
          const int64_t valid = jb.cols - c * 8;   // elements of this chunk inside the row
          if (valid < 8) {
            uint32_t w[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (e >= valid) w[e >> 1] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
            out = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        d[c] = out;
      }
    }
  }
}

}  // namespace gemm_tn_dev

namespace gemm_tn_impl {

cudaError_t launch_repack2(const RepackRequest* req, int num, int num_sms, cudaStream_t stream) {
  gemm_tn_dev::RepackArgs args{};
  int64_t rows = 0;
  int n = 0;
  for (int i = 0; i < num && n < 2; ++i) {
    if (req[i].rows <= 0) continue;
    args.job[n] = gemm_tn_dev::RepackJob{static_cast<const uint16_t*>(req[i].src), req[i].ld_src,
                                         static_cast<uint16_t*>(req[i].dst), req[i].ld_dst, req[i].rows,
                                         req[i].cols};
    rows += req[i].rows;
    ++n;
  }
  if (n == 0) return cudaSuccess;
  args.num_jobs = n;
  const int64_t max_grid = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
  const unsigned grid = static_cast<unsigned>(rows < max_grid ? rows : max_grid);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent_launch_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_tn_dev::repack_rows_kernel, args);
}

}  // namespace gemm_tn_impl
