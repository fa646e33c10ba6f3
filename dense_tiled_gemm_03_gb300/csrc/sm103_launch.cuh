// sm103_launch.cuh -- host-side launch helpers for one kernel configuration:
// per-device shared-memory opt-in, cluster launch, occupancy query.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "gemm_tn_internal.h"
#include "sm103_gemm_kernel.cuh"

namespace gemm_tn_impl {

template <class Cfg>
struct Launcher {
  static cudaError_t ensure_smem_attr() {
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done_mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(gemm_tn_dev::gemm_tn_sm103_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::kSmemBytes));
    if (e == cudaSuccess) done_mask.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  }

  static void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int grid, cudaStream_t stream,
                          bool dependent = false) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(gemm_tn_dev::kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (Cfg::kClusterSize > 1) {
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = Cfg::kClusterSize;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.numAttrs = 1;
    }
    if (dependent) {
      // programmatic dependent launch: the kernel's set-up may overlap the
      // previous kernel in the stream (the kernel waits before touching memory)
      attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
      ++cfg.numAttrs;
    }
  }

  static cudaError_t launch(const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
    cudaError_t e = ensure_smem_attr();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_config(cfg, attr, grid, stream, dependent_launch_enabled());
    return cudaLaunchKernelEx(&cfg, gemm_tn_dev::gemm_tn_sm103_kernel<Cfg>, args);
  }

  static int max_clusters() {
    if (ensure_smem_attr() != cudaSuccess) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (Cfg::kClusterSize == 1) {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_tn_dev::gemm_tn_sm103_kernel<Cfg>,
                                                        gemm_tn_dev::kNumThreads, Cfg::kSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return 0;
      }
      return per_sm * sms;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_config(cfg, attr, sms - sms % Cfg::kClusterSize, nullptr);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tn_dev::gemm_tn_sm103_kernel<Cfg>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return clusters;
  }
};

}  // namespace gemm_tn_impl
