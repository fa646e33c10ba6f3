// sm103_gemm_splitk.cu -- C = A x B^T split along K across the CTAs of a
// thread-block cluster, for problems with too few output tiles to occupy the
// GPU ("Tiling a matmul", section "Where it breaks": small M leaves little
// reuse and few tiles; split-K keeps all SMs busy).
//
// One cluster of S CTAs (S = 2, 4 or 8, on S SMs) owns one 128 x 128 output
// tile. CTA r of the cluster runs the usual TMA -> shared-memory ring ->
// tcgen05.mma pipeline over k-blocks [r * KB / S, (r + 1) * KB / S) into its
// own TMEM accumulator. The partial sums are then exchanged through
// distributed shared memory instead of global memory:
//   1. each CTA moves its fp32 accumulator TMEM -> registers -> its own shared
//      memory (the operand ring, idle once the last MMA has completed);
//   2. a cluster barrier makes every partial visible to the whole cluster;
//   3. CTA r adds, for rows [r * 128 / S, (r + 1) * 128 / S) of the tile, the
//      S partials in CTA order (ld.shared::cluster), rounds once to the output
//      type and stores those rows of C;
//   4. a second cluster barrier keeps every CTA's shared memory alive until
//      all peers have read it.
// The fixed order of the additions makes repeated launches bit-identical,
// and no global workspace, flag or atomic is involved.
//
// Every mbarrier wait is bounded (GEMM_TN_ERR_TIMEOUT through the status
// word); the roles never leave early, so every cluster barrier is always
// reached by every thread.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gemm_tn_internal.h"
#include "sm103_gemm_kernel.cuh"

namespace gemm_tn_dev {
namespace splitk {

constexpr int kThreads = 192;           // warp 0 TMA, warp 1 MMA, warps 2-5 TMEM drain; all reduce
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kBlockK = 64;             // one 128-byte swizzle row of 16-bit data
constexpr int kStages = 6;              // k-blocks the ring holds; kStages / kKb stages of kKb k-blocks
static_assert(kStages <= 32 && kStages % 2 == 0, "issued phases fit a 32-bit mask; stages of two k-blocks");
constexpr uint32_t kTileBytes = 128 * 64 * 2;                       // A or B box of one k-block
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kTileBytes;
constexpr uint32_t kRingEnd = kOffB + kStages * kTileBytes;        // 192 KiB
// fp32 partial tile, rows padded to 132 floats so that the 16-byte stores of
// one warp (32 rows, same column) spread over all banks
constexpr int kPartStride = kBlockN + 4;
constexpr uint32_t kPartBytes = kBlockM * kPartStride * 4;
constexpr uint32_t kOffBar = kRingEnd;                              // full[S], empty[S], acc_full, drain
constexpr int kNumBars = 2 * kStages + 2;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;                // + slack to align the base to 1024
constexpr uint32_t kTmemCols = 128;
static_assert(kPartBytes <= kRingEnd, "the partial tile fits in the idle operand ring");
static_assert(kSmemBytes <= 232448, "fits the opt-in shared memory of one CTA");

// What Watchdog needs to know of the launch.
template <int S>
struct ClusterOf {
  static constexpr int kClusterSize = S;
};

__device__ __forceinline__ float4 ld_shared_cluster_f4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kBf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

}  // namespace splitk

// kKb k-blocks per stage: with K a multiple of 64, one 3-D tensor copy moves
// two k-blocks of A or B ({64, 128, 2} boxes over {64, rows, K / 64} maps; the
// decode kernel below explains why), and the ring holds half as many stages
// of twice the size.
template <int S, bool kBf16, int kKb>
__global__ void __launch_bounds__(splitk::kThreads, 1) gemm_tn_splitk_kernel(const __grid_constant__ GemmArgs args) {
  using namespace splitk;
  static_assert(S == 2 || S == 4 || S == 8, "cluster of 2, 4 or 8 CTAs");
  static_assert(kKb == 1 || kKb == 2, "one or two k-blocks per stage");
  constexpr int kRing = kStages / kKb;          // stages in use
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t base = smem_addr(smem);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();          // this CTA's slice of K
  const int tile = static_cast<int>(blockIdx.x) / S;
  const int tn = args.div_m_tiles.div(tile);
  const int tm = tile - tn * args.num_m_tiles;
  // this CTA's stages: [kb0, kb1) in units of kKb k-blocks
  const int units = (args.num_k_blocks + kKb - 1) / kKb;
  const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * units / S);
  const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * units / S);

  auto a_tile = [&](int s) { return base + kOffA + s * kKb * kTileBytes; };
  auto b_tile = [&](int s) { return base + kOffB + s * kKb * kTileBytes; };
  auto full_bar = [&](int s) { return base + kOffBar + 8u * s; };
  auto empty_bar = [&](int s) { return base + kOffBar + 8u * (kStages + s); };
  const uint32_t acc_full_bar = base + kOffBar + 8u * (2 * kStages);
  const uint32_t drain_bar = acc_full_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffAbort);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_full_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_descriptor(&args.tmap_a);
    tma_prefetch_descriptor(&args.tmap_b);
  }
  if (warp == 1) {
    tmem_alloc<1>(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish<1>();
  }
  // The pipeline uses only this CTA's barriers and TMEM, so set-up ends at a
  // CTA barrier. Its peers' shared memory is touched only in the reduction
  // (and by a role that gives up, after the watchdog's budget): the cluster
  // barrier that guarantees every peer has started is arrived at here and
  // waited for there, off the path to the first copy.
  tc_fence_before_sync();
  __syncthreads();
  cluster_arrive_relaxed();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // set-up may overlap the previous kernel in the stream; memory waits for
  // it: the producer just before its first copy, every other thread here
  if (warp != 0 || lane != 0) {
    griddep_wait();
    griddep_launch_dependents();
  }
  const Watchdog<ClusterOf<S>> wd{&args, abort_flag, smem_addr(const_cast<uint32_t*>(abort_flag))};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      IssuedPhases issued;
      bool dep_waited = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wd.wait(empty_bar(stage), phase ^ 1u)) break;
        if (!dep_waited) {
          griddep_wait();
          griddep_launch_dependents();
          dep_waited = true;
        }
        const uint32_t fb = full_bar(stage);
        mbar_arrive_expect_tx(fb, 2 * kKb * kTileBytes);
        if (kb - kb0 != args.drop_load_kb) {
          if constexpr (kKb == 2) {
            tma_load_3d(&args.tmap_a, a_tile(stage), fb, 0, tm * kBlockM, 2 * kb);
            tma_load_3d(&args.tmap_b, b_tile(stage), fb, 0, tn * kBlockN, 2 * kb);
          } else {
            tma_load_2d(&args.tmap_a, a_tile(stage), fb, kb * kBlockK, tm * kBlockM);
            tma_load_2d(&args.tmap_b, b_tile(stage), fb, kb * kBlockK, tn * kBlockN);
          }
        }
        issued.record(stage, phase);
        if (++stage == kRing) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!dep_waited) {
        griddep_wait();
        griddep_launch_dependents();
      }
      // loads still landing after another role gave up finish before exit
      for (int s = 0; s < kRing; ++s)
        if (issued.any(s)) wd.drain(full_bar(s), issued.phase(s));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdesc = mma_idesc_f16(kBf16, kBlockM, kBlockN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wd.wait(full_bar(stage), phase)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kKb * (kBlockK / 16); ++kk) {
          // k-block kk / 4 of the stage, 16-element step kk % 4 within it
          const uint64_t a_desc = sw128_kmajor_desc(a_tile(stage) + (kk >> 2) * kTileBytes);
          const uint64_t b_desc = sw128_kmajor_desc(b_tile(stage) + (kk >> 2) * kTileBytes);
          mma_f16<1>(tmem_base, a_desc + 2u * (kk & 3), b_desc + 2u * (kk & 3), kIdesc,
                     (kb > kb0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(empty_bar(stage));
        if (++stage == kRing) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) mma_commit(acc_full_bar);
      // every MMA issued here completes before TMEM is freed
      mma_commit(drain_bar);
      wd.drain(drain_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- TMEM -> own shared memory
    const uint32_t quarter = warp & 3u;          // TMEM lanes this warp may read
    const bool ok = __all_sync(0xffffffffu, wd.wait(acc_full_bar, 0));
    if (ok) {
      tc_fence_after_sync();
      const uint32_t row = quarter * 32u + lane;
      const uint32_t t_row = tmem_base + ((quarter * 32u) << 16);
#pragma unroll 1
      for (int chunk = 0; chunk < kBlockN / 32; ++chunk) {
        uint32_t r[32];
        tmem_load_32x32(t_row + static_cast<uint32_t>(chunk * 32), r);
        tmem_load_wait();
        const uint32_t dst = base + (row * kPartStride + chunk * 32) * 4u;
#pragma unroll
        for (int j = 0; j < 8; ++j) st_shared_v4(dst + 16u * j, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
      }
    }
  }
  __syncwarp();

  // ---------------------------------------------------------------- cluster reduction
  // every peer has started (the set-up's arrival); then every CTA's partial
  // is in its shared memory: make them visible cluster-wide
  cluster_wait();
  tc_fence_before_sync();
  cluster_sync_all();
  {
    constexpr int kRows = kBlockM / S;                        // rows of the tile this CTA finishes
    constexpr int kPositions = kRows * (kBlockN / 4);         // float4 positions of those rows
    // A shared::cluster load is a round trip over the cluster's network:
    // each thread issues the loads of kBatch positions (16 float4 loads for
    // every S) before it adds and stores any of them, instead of one position
    // per round trip (1024^3: the reduction 2.3 -> 1.8 us). The network's
    // bandwidth, ~17 bytes per SM clock here, bounds the rest; pushing the
    // peers' rows with bulk copies into local shared memory instead was no
    // faster at S = 2 and slower at S = 4 and 8.
    constexpr int kBatch = 16 / S;
    const int r0 = static_cast<int>(rank) * kRows;
    uint16_t* cbase = static_cast<uint16_t*>(args.c);
    for (int first = threadIdx.x; first < kPositions; first += kThreads * kBatch) {
      float4 v[kBatch][S];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int idx = first + u * kThreads;
        if (idx < kPositions) {
          const int row = r0 + (idx >> 5);
          const int col = (idx & 31) * 4;
          const uint32_t off = base + static_cast<uint32_t>(row * kPartStride + col) * 4u;
#pragma unroll
          for (int s = 0; s < S; ++s) v[u][s] = ld_shared_cluster_f4(map_to_cta(off, static_cast<uint32_t>(s)));
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int idx = first + u * kThreads;
        if (idx >= kPositions) break;
        const int row = r0 + (idx >> 5);
        const int col = (idx & 31) * 4;
        float4 acc = v[u][0];
#pragma unroll
        for (int s = 1; s < S; ++s) {   // CTA order: the same sum on every launch
          acc.x += v[u][s].x;
          acc.y += v[u][s].y;
          acc.z += v[u][s].z;
          acc.w += v[u][s].w;
        }
        const int grow = tm * kBlockM + row;
        const int gcol = tn * kBlockN + col;
        if (grow >= args.m || gcol >= args.n) continue;
        uint16_t* dst = cbase + static_cast<int64_t>(grow) * args.ldc + gcol;
        const uint32_t lo = pack2<kBf16>(acc.x, acc.y), hi = pack2<kBf16>(acc.z, acc.w);
        if (gcol + 4 <= args.n && (reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
        } else {
          const uint16_t e[4] = {static_cast<uint16_t>(lo & 0xFFFFu), static_cast<uint16_t>(lo >> 16),
                                 static_cast<uint16_t>(hi & 0xFFFFu), static_cast<uint16_t>(hi >> 16)};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (gcol + j < args.n) dst[j] = e[j];
        }
      }
    }
  }
  // peers may still be reading this CTA's partial
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<1>(tmem_base, kTmemCols);
  }
}

}  // namespace gemm_tn_dev

namespace gemm_tn_dev {
namespace decode {

// Few rows of A (decode-like M <= 32): the roles swap. 128 rows of B are the
// MMA's M side and A's kN rows (zero-filled past M) its N side, so the
// accumulator holds C^T for 128 columns of C. A stage then carries 16 KiB of B
// and only kN * 128 bytes of A per k-block, and about twice the B bytes of the
// 128 x 128 split-K kernel are in flight per SM.
//
// kKb k-blocks per stage: with K a multiple of 64, one 3-D tensor copy moves
// two k-blocks of B, and another two of A, at once ({64, rows, 2} boxes over
// the maps {64, rows, K / 64}; a k-block past K, when their count is odd,
// reads as zeros). The producer thread issues half the copies and barrier operations
// per byte: at 16 k-blocks per CTA its issue rate, ~550 clocks per k-block,
// had paced the stream (8 x 4096 x 4096: 6.26 -> 5.73 us per call replayed).
constexpr int kThreads = 192;
constexpr uint32_t kBTileBytes = 128 * 64 * 2;
constexpr uint32_t kRingBudget = 200 * 1024;

template <int kN, int kKb>
struct Layout {
  static constexpr uint32_t kATileBytes = kN * 64 * 2;                   // A of one k-block
  static constexpr uint32_t kStageB = kKb * kBTileBytes;                 // B of one stage
  static constexpr uint32_t kStageA = kKb * kATileBytes;                 // A of one stage
  static constexpr int kStages = static_cast<int>(kRingBudget / (kStageB + kStageA));
  static_assert(kKb == 1 || kKb == 2, "one or two k-blocks per stage");
  static_assert(kStages >= 1 && kStages <= 32, "issued phases fit a 32-bit mask");
  static constexpr uint32_t kOffB = 0;
  static constexpr uint32_t kOffA = kOffB + kStages * kStageB;
  static constexpr uint32_t kRingEnd = kOffA + kStages * kStageA;
  static constexpr int kPartStride = kN + 4;                            // floats per partial row (n)
  static constexpr uint32_t kPartBytes = 128 * kPartStride * 4;
  static constexpr uint32_t kOffBar = kRingEnd;                          // full[S], empty[S], acc_full, drain
  static constexpr int kNumBars = 2 * kStages + 2;
  static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
  static constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;
  static constexpr uint32_t kTmemCols = kN < 32 ? 32 : kN;
  static_assert(kN == 16 || kN == 32, "A rows per MMA: 16 or 32");
  static_assert(kATileBytes % 1024 == 0 && kBTileBytes % 1024 == 0, "swizzle atoms stay 1024-aligned");
  static_assert(kPartBytes <= kRingEnd, "the partial tile fits in the idle ring");
  static_assert(kSmemBytes <= 214 * 1024 + 256, "no more shared memory than the other GEMM kernels");
};

}  // namespace decode

template <int S, int kN, bool kBf16, int kKb>
__global__ void __launch_bounds__(decode::kThreads, 1) gemm_tn_decode_kernel(const __grid_constant__ GemmArgs args) {
  using L = decode::Layout<kN, kKb>;
  static_assert(S == 2 || S == 4 || S == 8, "cluster of 2, 4 or 8 CTAs");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t base = smem_addr(smem);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();          // this CTA's slice of K
  const int tn = static_cast<int>(blockIdx.x) / S;  // 128 columns of C (rows of B)
  // this CTA's stages: [kb0, kb1) in units of kKb k-blocks
  const int units = (args.num_k_blocks + kKb - 1) / kKb;
  const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * units / S);
  const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * units / S);

  auto b_tile = [&](int s) { return base + L::kOffB + s * L::kStageB; };
  auto a_tile = [&](int s) { return base + L::kOffA + s * L::kStageA; };
  auto full_bar = [&](int s) { return base + L::kOffBar + 8u * s; };
  auto empty_bar = [&](int s) { return base + L::kOffBar + 8u * (L::kStages + s); };
  const uint32_t acc_full_bar = base + L::kOffBar + 8u * (2 * L::kStages);
  const uint32_t drain_bar = acc_full_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kOffAbort);

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_full_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_descriptor(&args.tmap_a);
    tma_prefetch_descriptor(&args.tmap_b);
  }
  if (warp == 1) {
    tmem_alloc<1>(smem_addr(tmem_slot), L::kTmemCols);
    tmem_relinquish<1>();
  }
  // The pipeline uses only this CTA's barriers and TMEM, so set-up ends at a
  // CTA barrier. Its peers' shared memory is touched only in the reduction
  // (and by a role that gives up, after the watchdog's budget): the cluster
  // barrier that guarantees every peer has started is arrived at here and
  // waited for there, off the path to the first copy.
  tc_fence_before_sync();
  __syncthreads();
  cluster_arrive_relaxed();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // set-up may overlap the previous kernel in the stream; memory waits for
  // it: the producer just before its first copy, every other thread here
  if (warp != 0 || lane != 0) {
    griddep_wait();
    griddep_launch_dependents();
  }
  const Watchdog<splitk::ClusterOf<S>> wd{&args, abort_flag, smem_addr(const_cast<uint32_t*>(abort_flag))};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      IssuedPhases issued;
      bool dep_waited = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wd.wait(empty_bar(stage), phase ^ 1u)) break;
        if (!dep_waited) {
          griddep_wait();
          griddep_launch_dependents();
          dep_waited = true;
        }
        const uint32_t fb = full_bar(stage);
        mbar_arrive_expect_tx(fb, L::kStageB + L::kStageA);
        if (kb - kb0 != args.drop_load_kb) {
          if constexpr (kKb == 2) {
            tma_load_3d(&args.tmap_b, b_tile(stage), fb, 0, tn * 128, 2 * kb);
            tma_load_3d(&args.tmap_a, a_tile(stage), fb, 0, 0, 2 * kb);   // rows past M read as zero
          } else {
            tma_load_2d(&args.tmap_b, b_tile(stage), fb, kb * 64, tn * 128);
            tma_load_2d(&args.tmap_a, a_tile(stage), fb, kb * 64, 0);   // rows past M read as zero
          }
        }
        issued.record(stage, phase);
        if (++stage == L::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!dep_waited) {
        griddep_wait();
        griddep_launch_dependents();
      }
      for (int s = 0; s < L::kStages; ++s)
        if (issued.any(s)) wd.drain(full_bar(s), issued.phase(s));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer: D[n][m] += B[n][k] A[m][k]
      constexpr uint32_t kIdesc = mma_idesc_f16(kBf16, 128, kN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wd.wait(full_bar(stage), phase)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 4 * kKb; ++kk) {
          // k-block kk / 4 of the stage, 16-element step kk % 4 within it
          const uint64_t b_desc = sw128_kmajor_desc(b_tile(stage) + (kk >> 2) * decode::kBTileBytes);
          const uint64_t a_desc = sw128_kmajor_desc(a_tile(stage) + (kk >> 2) * L::kATileBytes);
          mma_f16<1>(tmem_base, b_desc + 2u * (kk & 3), a_desc + 2u * (kk & 3), kIdesc,
                     (kb > kb0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(empty_bar(stage));
        if (++stage == L::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) mma_commit(acc_full_bar);
      mma_commit(drain_bar);
      wd.drain(drain_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- TMEM -> own shared memory
    const uint32_t quarter = warp & 3u;
    const bool ok = __all_sync(0xffffffffu, wd.wait(acc_full_bar, 0));
    if (ok) {
      tc_fence_after_sync();
      const uint32_t row = quarter * 32u + lane;   // column n of this 128-column block
      const uint32_t t_row = tmem_base + ((quarter * 32u) << 16);
      const uint32_t dst = base + row * L::kPartStride * 4u;
      if constexpr (kN == 16) {
        uint32_t r[16];
        tmem_load_32x16(t_row, r);
        tmem_load_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j) st_shared_v4(dst + 16u * j, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
      } else {
#pragma unroll 1
        for (int chunk = 0; chunk < kN / 32; ++chunk) {
          uint32_t r[32];
          tmem_load_32x32(t_row + static_cast<uint32_t>(chunk * 32), r);
          tmem_load_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(dst + 128u * chunk + 16u * j, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        }
      }
    }
  }
  __syncwarp();

  // ---------------------------------------------------------------- cluster reduction
  cluster_wait();   // every peer has started (the set-up's arrival)
  tc_fence_before_sync();
  cluster_sync_all();
  {
    constexpr int kRows = 128 / S;          // columns of C (rows of the partial) this CTA finishes
    const int r0 = static_cast<int>(rank) * kRows;
    uint16_t* cbase = static_cast<uint16_t*>(args.c);
    for (int idx = threadIdx.x; idx < kRows * (kN / 4); idx += decode::kThreads) {
      const int nl = r0 + idx % kRows;       // consecutive threads: consecutive columns of C
      const int m0 = (idx / kRows) * 4;
      const int gn = tn * 128 + nl;
      if (gn >= args.n || m0 >= args.m) continue;
      const uint32_t off = base + static_cast<uint32_t>(nl * L::kPartStride + m0) * 4u;
      float4 v[S];
#pragma unroll
      for (int s = 0; s < S; ++s) v[s] = splitk::ld_shared_cluster_f4(map_to_cta(off, static_cast<uint32_t>(s)));
      float4 acc = v[0];
#pragma unroll
      for (int s = 1; s < S; ++s) {   // CTA order: the same sum on every launch
        acc.x += v[s].x;
        acc.y += v[s].y;
        acc.z += v[s].z;
        acc.w += v[s].w;
      }
      const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (m0 + j < args.m)
          cbase[static_cast<int64_t>(m0 + j) * args.ldc + gn] =
              static_cast<uint16_t>(splitk::pack2<kBf16>(vals[j], 0.0f) & 0xFFFFu);
    }
  }
  // peers may still be reading this CTA's partial
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<1>(tmem_base, L::kTmemCols);
  }
}

}  // namespace gemm_tn_dev
namespace gemm_tn_impl {
namespace {

template <int S, bool kBf16, int kKb>
struct SplitKLauncher {
  static cudaError_t ensure_smem_attr() {
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done_mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(gemm_tn_dev::gemm_tn_splitk_kernel<S, kBf16, kKb>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(gemm_tn_dev::splitk::kSmemBytes));
    if (e == cudaSuccess) done_mask.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  }

  static void fill(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int grid, cudaStream_t stream, bool dep) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(gemm_tn_dev::splitk::kThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_tn_dev::splitk::kSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dep) {
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.numAttrs = 2;
    }
  }

  static cudaError_t launch(const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
    cudaError_t e = ensure_smem_attr();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill(cfg, attr, grid, stream, dependent_launch_enabled());
    return cudaLaunchKernelEx(&cfg, gemm_tn_dev::gemm_tn_splitk_kernel<S, kBf16, kKb>, args);
  }

  static int max_clusters(int num_sms) {
    if (ensure_smem_attr() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill(cfg, attr, num_sms - num_sms % S, nullptr, false);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tn_dev::gemm_tn_splitk_kernel<S, kBf16, kKb>, &cfg) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return clusters;
  }
};

template <int S, int kN, bool kBf16, int kKb>
struct DecodeLauncher {
  static cudaError_t launch(const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
    using L = gemm_tn_dev::decode::Layout<kN, kKb>;
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done_mask.load(std::memory_order_acquire) & bit)) {
      e = cudaFuncSetAttribute(gemm_tn_dev::gemm_tn_decode_kernel<S, kN, kBf16, kKb>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kSmemBytes));
      if (e != cudaSuccess) return e;
      done_mask.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(gemm_tn_dev::decode::kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dependent_launch_enabled()) {
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, gemm_tn_dev::gemm_tn_decode_kernel<S, kN, kBf16, kKb>, args);
  }
};

template <int kN, bool kBf16, int kKb>
cudaError_t launch_decode_split(int splits, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
  switch (splits) {
    case 2: return DecodeLauncher<2, kN, kBf16, kKb>::launch(args, grid, stream);
    case 4: return DecodeLauncher<4, kN, kBf16, kKb>::launch(args, grid, stream);
    case 8: return DecodeLauncher<8, kN, kBf16, kKb>::launch(args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int kN, bool kBf16>
cudaError_t launch_decode_rows(int splits, bool k_pairs, const gemm_tn_dev::GemmArgs& args, int grid,
                               cudaStream_t stream) {
  return k_pairs ? launch_decode_split<kN, kBf16, 2>(splits, args, grid, stream)
                 : launch_decode_split<kN, kBf16, 1>(splits, args, grid, stream);
}

}  // namespace

// Rows of A per MMA of the decode kernel for an M-row problem (0: M > 32).
// With 33-64 rows the 128 x 128 split-K kernel measured as fast or faster
// (64 x 2048 x 8192: 12.1 against 12.6 us): C's column-wise stores cost more.
int decode_rows(int64_t m) { return m <= 16 ? 16 : m <= 32 ? 32 : 0; }

cudaError_t launch_gemm_decode(int splits, int rows, bool bf16, bool k_pairs, const gemm_tn_dev::GemmArgs& args,
                               int grid, cudaStream_t stream) {
  switch (rows) {
    case 16: return bf16 ? launch_decode_rows<16, true>(splits, k_pairs, args, grid, stream)
                         : launch_decode_rows<16, false>(splits, k_pairs, args, grid, stream);
    case 32: return bf16 ? launch_decode_rows<32, true>(splits, k_pairs, args, grid, stream)
                         : launch_decode_rows<32, false>(splits, k_pairs, args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <bool kBf16, int kKb>
cudaError_t launch_splitk_kb(int splits, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream) {
  switch (splits) {
    case 2: return SplitKLauncher<2, kBf16, kKb>::launch(args, grid, stream);
    case 4: return SplitKLauncher<4, kBf16, kKb>::launch(args, grid, stream);
    case 8: return SplitKLauncher<8, kBf16, kKb>::launch(args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_splitk(int splits, bool bf16, bool k_pairs, const gemm_tn_dev::GemmArgs& args, int grid,
                               cudaStream_t stream) {
  if (bf16) return k_pairs ? launch_splitk_kb<true, 2>(splits, args, grid, stream)
                           : launch_splitk_kb<true, 1>(splits, args, grid, stream);
  return k_pairs ? launch_splitk_kb<false, 2>(splits, args, grid, stream)
                 : launch_splitk_kb<false, 1>(splits, args, grid, stream);
}

// (both forms of a stage take the same shared memory and threads)
int max_resident_splitk(int splits, bool bf16, int num_sms) {
  switch (splits) {
    case 2: return bf16 ? SplitKLauncher<2, true, 1>::max_clusters(num_sms)
                        : SplitKLauncher<2, false, 1>::max_clusters(num_sms);
    case 4: return bf16 ? SplitKLauncher<4, true, 1>::max_clusters(num_sms)
                        : SplitKLauncher<4, false, 1>::max_clusters(num_sms);
    case 8: return bf16 ? SplitKLauncher<8, true, 1>::max_clusters(num_sms)
                        : SplitKLauncher<8, false, 1>::max_clusters(num_sms);
    default: return 0;
  }
}

}  // namespace gemm_tn_impl
