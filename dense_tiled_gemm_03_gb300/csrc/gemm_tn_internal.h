// gemm_tn_internal.h -- host-side interface between the C-ABI translation unit
// and the translation units that hold the kernel instantiations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace gemm_tn_dev {
struct GemmArgs;

// Kernel arguments of the attention forward pass (sm103_flash_attn.cu).
struct FlashArgs {
  CUtensorMap tmap_q;   // 3-D {heads * dim, seq, batch} maps, boxes {64, 128, 1},
  CUtensorMap tmap_k;   // 128-byte swizzle, zero fill past seq
  CUtensorMap tmap_v;
  void* o;              // [batch, seq, heads, dim], 16-byte aligned
  int batch, seq, heads;
  int num_q_tiles;      // CTAs per (batch, head): ceil(seq / flash_attn_rows_per_cta())
  int head_group;       // (batch, head) pairs whose query tiles run interleaved
  float scale_log2;     // softmax scale * log2(e), > 0
  int causal;
  int* status;          // optional device status word (watchdog)
  uint64_t timeout_ns;
  int drop_load_block;  // test hook: key tile whose K load the first CTA skips (-1: none)
};
}  // namespace gemm_tn_dev

namespace gemm_tn_impl {

// Frozen configuration table ("TileLang: a tile language one level below
// Triton", section "A few engineering points": freeze tuning results into a
// table). Index order is part of the ABI (gemm_tn_config_name).
enum ConfigId : int {
  kCfg1CtaN256 = 0,   // one CTA per 128 x 256 tile, 4-stage ring
  kCfg1CtaN128 = 1,   // one CTA per 128 x 128 tile, 6-stage ring (skinny / few tiles)
  kCfg2CtaN256 = 2,   // CTA pair per 256 x 256 tile (cta_group::2), 6-stage ring
  kCfg2CtaN128 = 3,   // CTA pair per 256 x 128 tile (cta_group::2), 8-stage ring
  kCfg2CtaN256Mc = 4, // 4-CTA cluster: two pairs on 256 x 512, A shared by TMA multicast
  kCfg1CtaSplitK = 5, // 128 x 128 tiles, K split over a cluster of 2, 4 or 8 CTAs (few tiles, long K)
  kCfgDecodeSplitK = 6, // M <= 32: B's rows on the MMA's M side, K split over a cluster (decode-like)
  kCfg1CtaN64 = 7,    // one CTA per 128 x 64 tile, 8-stage ring (small problems: more SMs share the loads)
  kNumConfigs = 8
};

struct ConfigInfo {
  const char* name;
  int cta_group;
  int tile_m;        // rows per tile (128 * cta_group)
  int block_n;       // columns per tile (per CTA pair)
  int b_rows;        // rows of B one CTA loads (block_n / cta_group)
  int stages;
  int cluster_pairs; // CTA pairs per cluster (2: A shared by multicast)
  int a_box_rows;    // rows of A one TMA load brings (64 with multicast halves)
};

const ConfigInfo& config_info(int id);

// Launch one configuration. grid = CTAs (a multiple of cta_group).
cudaError_t launch_gemm(int id, bool bf16, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream);

// Co-resident clusters (CTA pairs, or single CTAs) of a configuration on the
// current device; 0 on error.
int max_resident_clusters(int id, bool bf16);

// Row repack of one matrix: dst[r][0:ld_dst] = src[r][0:cols] padded with
// zeros, for r < rows (ld_dst a multiple of 8, dst 16-byte aligned).
struct RepackRequest {
  const void* src;
  int64_t ld_src;
  void* dst;
  int64_t ld_dst;
  int64_t rows;
  int64_t cols;
};

// Attention forward pass: one CTA per flash_attn_rows_per_cta() queries of
// one (batch, head); grid = num_q_tiles * batch * heads. head_dim 64 or 128.
int flash_attn_rows_per_cta();
cudaError_t launch_flash_attn(int head_dim, bool bf16, const gemm_tn_dev::FlashArgs& args, unsigned grid,
                              cudaStream_t stream);

// Whether the GEMM and repack kernels are launched as programmatic dependents
// of the previous kernel in their stream (on unless GEMM_TN_PDL=0).
bool dependent_launch_enabled();

// One launch repacking up to two matrices (entries with rows <= 0 are skipped).
cudaError_t launch_repack2(const RepackRequest* req, int num, int num_sms, cudaStream_t stream);

}  // namespace gemm_tn_impl
