// sm103_gemm_kernel.cuh -- the persistent, warp-specialized tcgen05 GEMM kernel
// for C[M,N] = A[M,K] x B[N,K]^T on sm_103a (GB300).
//
// Structure (prior art on the pages, redesigned for tcgen05 / TMEM):
//  * Block tiling: each CTA (or CTA pair) owns output tiles and walks K in
//    64-element blocks ("0. A Minimal Hopper Matmul", section "Block Tiling";
//    "Tiling a matmul", section "Counting traffic").
//  * A multi-stage shared-memory ring filled by TMA and handed off through
//    full/empty mbarriers ("Tiling a matmul", section "Pipelining";
//    "TileLang: a tile language one level below Triton", section "What it
//    generated": 3 full + 3 empty barriers around a TMA producer).
//  * Warp specialization: warp 0 is the TMA producer, one thread of warp 1
//    issues every tcgen05.mma, warps 2..9 are the epilogue (two per 32-lane
//    quarter of TMEM, on alternate 32-column chunks).
//  * Accumulators live in tensor memory (TMEM), double-buffered so the
//    epilogue of one tile overlaps the main loop of the next. The operand
//    round trip through registers that the Hopper V0 kernel pays ("0. A
//    Minimal Hopper Matmul", sections "Data Flow" and "What's Next") does not
//    exist here: tcgen05.mma reads both operands from shared memory.
//  * Persistent scheduler with grouped rasterization so tiles running at the
//    same time share rows of A and of B in L2 ("Tiling a matmul", section "The
//    levels of tiling", and "Check yourself" on launch order).
//  * kCtaGroup == 2: a cluster of two CTAs on two SMs computes a 256-row tile
//    with cta_group::2 MMAs; each CTA loads its own 128 rows of A and half of
//    the B tile, and the pair's leader issues the MMAs.
//  * Ragged M/N/K: TMA zero-fills out-of-range boxes; the epilogue stores
//    only in-range elements, which also handles any row stride of C.
//  * Barriers sit after every TMA/MMA buffer in a fixed layout ("0. A Minimal
//    Hopper Matmul", section "Epilogue": a barrier placed inside a live TMA
//    destination corrupts results).
//  * Every wait is bounded: past the deadline the kernel records
//    GEMM_TN_ERR_TIMEOUT, tells the other roles to stop, drains its own async
//    work, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace gemm_tn_dev {

constexpr int kNumThreads = 320;       // 10 warps
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kFirstEpilogueWarp = 2;
// two epilogue warps per 32-lane quarter of TMEM, on alternate 32-column
// chunks: a chunk is a chain of short dependent steps (TMEM load, convert,
// staging stores, proxy fence, TMA store), so two chains per quarter halve
// the epilogue that is left exposed after a CTA's last tile
constexpr int kNumEpilogueWarps = 8;
constexpr int kStatusTimeout = 6;      // == GEMM_TN_ERR_TIMEOUT

// Division by an invariant divisor d (1 <= d < 2^31) as a multiply-high, an
// add and a shift, exact for every dividend n < 2^31: Granlund and
// Montgomery, "Division by invariant integers using multiplication" (1994),
// the round-up method. With l = ceil(log2 d) and
// mul = floor(2^32 (2^l - d) / d) + 1 (below 2^32), floor(n / d) =
// (umulhi(n, mul) + n) >> l; the sum stays below 2^32 since umulhi(n, mul) < n.
// A runtime 32-bit division is a dependent chain of ~20 instructions through
// the reciprocal unit, on the producer's path to its first copy.
struct FastDiv {
  uint32_t mul;
  uint32_t shift;
#ifdef __CUDACC__
  __device__ __forceinline__ int div(int n) const {
    const uint32_t u = static_cast<uint32_t>(n);
    return static_cast<int>((__umulhi(u, mul) + u) >> shift);
  }
#endif
};

// Kernel arguments. Tensor maps first: they must be 64-byte aligned.
struct GemmArgs {
  CUtensorMap tmap_a;     // A: dims {K, M}, box {64, 128}, 128B swizzle
  CUtensorMap tmap_b;     // B: dims {K, N}, box {64, BN / cta_group}, 128B swizzle
  CUtensorMap tmap_c;     // C: dims {N, M}, box {32, 32}, 64B swizzle (valid when c_tma_store)
  CUtensorMap tmap_b_split;  // B with box rows BN / cta_group / split (valid when split > 1)
  void* c;                // C [M, N], row stride ldc elements
  int64_t ldc;
  int32_t c_tma_store;    // 1: epilogue stores through the TMA; 0: predicated element stores
  int32_t m, n, k;
  int32_t num_m_tiles, num_n_tiles, num_k_blocks, num_tiles;
  int32_t group_m;        // tile rows per rasterization group
  FastDiv div_group;      // by group_m * num_n_tiles (tiles per group)
  FastDiv div_rows;       // by group_m
  FastDiv div_last_rows;  // by the tile rows of the last group (num_m_tiles - its first row)
  FastDiv div_m_tiles;    // by num_m_tiles (the split-K and decode kernels' column-major tile order)
  int* status;            // nullable device int: first error code wins
  uint64_t timeout_ns;    // per-wait watchdog budget
  int32_t drop_load_kb;   // test hook: the producer skips the loads of this stage of its first unit of
                          // work (a stage holds one k-block, or two with kKPairs and in the split-K and
                          // decode kernels); -1: never
  // Work split over the num_workers clusters of the grid. Tiles [0, dp_tiles)
  // go whole and round-robin to the workers. The sk_iters k-block iterations
  // of tiles [dp_tiles, num_tiles) (stream-K tail) are cut into sk_workers
  // contiguous ranges, one for each of workers 0 .. sk_workers - 1; a tile cut
  // between workers is finished by the worker holding its first k-block,
  // which adds the others' fp32 partials.
  int32_t dp_tiles;
  int32_t num_workers;
  int64_t sk_iters;
  int32_t sk_workers;
  // Tail split: tiles [split_begin, num_tiles) -- the last, partial wave --
  // are each cut into `split` sub-tiles of block_n / split columns, so that
  // wave holds more, shorter units of work (split 1: no cut).
  int32_t split;
  int32_t split_log2;     // log2(split)
  int32_t split_begin;
  int32_t dp_units;       // split_begin + (dp_tiles - split_begin) * split
  // Fused epilogue (kFused kernels): D = act(alpha * acc + beta * C + bias[j]),
  // stored in C's element type out_kind: 0 the input dtype, 1 fp32, 2 fp8
  // e4m3 (round to nearest even, saturating at +-448).
  float alpha, beta;
  const float* bias;      // nullable [N]
  int32_t activation;     // 0 none, 1 relu, 2 gelu
  int32_t out_kind;
  float* partials;        // per CTA: block_n / 32 chunks x 8 x 128 rows of float4 (stream-K only)
  uint64_t* flags;        // per CTA and epilogue warp: flag_epoch once its partial rows are written
  uint64_t flag_epoch;    // this launch's flag value (unique per launch; stale values never match)
  // Memory-bound problems with one row of tiles (B streamed once, A re-read
  // from L2): k_rotate != 0 starts every tile that covers all of K at its
  // own k-block (k_start) and wraps around, and b_evict_first marks the B
  // loads evict-first in L2.
  int32_t k_rotate;
  int32_t b_evict_first;
};

template <int kCtaGroup_, int kBlockN_, int kStages_, bool kBf16_, int kClusterPairs_ = 1, bool kBMnMajor_ = false,
          bool kFused_ = false, bool kTailSplit_ = false, bool kKPairs_ = false>
struct GemmConfig {
  static constexpr int kCtaGroup = kCtaGroup_;
  // kKPairs: a stage holds two k-blocks, moved by one 3-D tensor copy per
  // operand ({64, rows, 2} boxes over {64, rows, K / 64} maps; a k-block past
  // K reads as zeros), for single-CTA tiles whose units of work each cover all
  // of K in order (no stream-K range, rotated K walk or cut tail tile). The
  // producer then issues half the copies and barrier operations per byte.
  static constexpr bool kKPairs = kKPairs_;
  static constexpr int kKb = kKPairs ? 2 : 1;   // k-blocks per stage
  static constexpr bool kFused = kFused_;
  // kTailSplit: the instantiation that can run the cut sub-tiles of the last
  // wave; the others keep every unit a whole tile (the split arithmetic
  // measurably slows the main loops when compiled in but unused).
  static constexpr bool kTailSplit = kTailSplit_;
  // kBMnMajor: B is stored [K, N] with N contiguous (C = A x B), loaded in
  // 64 x 64 boxes and read by the MMA through MN-major descriptors.
  static constexpr bool kBMnMajor = kBMnMajor_;
  static constexpr uint32_t kBMnBoxBytes = 64 * 64 * 2;
  // kClusterPairs == 2: a cluster of two CTA pairs side by side along N that
  // share their rows of A. Each CTA loads one 64-row half of its A block and
  // TMA-multicasts it to the CTA at the same position in the other pair.
  static constexpr int kClusterPairs = kClusterPairs_;
  static constexpr bool kMulticastA = kClusterPairs == 2;
  static constexpr int kClusterSize = kCtaGroup * kClusterPairs;
  static constexpr int kClusterN = kBlockN_ * kClusterPairs;   // output columns per cluster
  static constexpr int kBlockM = 128;                    // rows per CTA
  static constexpr int kTileM = kBlockM * kCtaGroup;     // rows per tile (MMA M)
  static constexpr int kBlockN = kBlockN_;               // columns per tile (MMA N)
  static constexpr int kBRows = kBlockN / kCtaGroup;     // rows of B each CTA loads
  static constexpr int kBlockK = 64;                     // one 128-byte swizzle row of 16-bit data
  static constexpr int kMmaK = 16;
  static constexpr int kStages = kStages_;
  static constexpr bool kBf16 = kBf16_;
  static constexpr uint32_t kATileBytes = kBlockM * kBlockK * 2;   // A of one k-block
  static constexpr uint32_t kBTileBytes = kBRows * kBlockK * 2;     // B of one k-block
  static constexpr uint32_t kStageA = kKb * kATileBytes;            // A of one stage
  static constexpr uint32_t kStageB = kKb * kBTileBytes;            // B of one stage
  static constexpr int kAccCols = kBlockN;               // fp32 columns per accumulator
  static constexpr int kNumAcc = 2;
  static constexpr uint32_t kTmemCols = kAccCols * kNumAcc;
  // epilogue staging, per warp: either 32 rows x (16 packed words + 1 pad
  // word) for the transposed element stores, or two 32 x 32 16-bit boxes
  // (2 KiB each, 64-byte swizzle) for the TMA store
  static constexpr int kStageRowWords = 17;
  static constexpr uint32_t kEpiWarpBytes = 4096;
  static constexpr uint32_t kEpiBytes = kNumEpilogueWarps * kEpiWarpBytes;
  static_assert(32 * kStageRowWords * 4 <= kEpiWarpBytes, "transpose staging fits the warp's slot");
  // layout (offsets from the 1024-aligned base)
  static constexpr uint32_t kOffA = 0;
  static constexpr uint32_t kOffB = kOffA + kStages * kStageA;
  static constexpr uint32_t kOffEpi = kOffB + kStages * kStageB;
  static constexpr uint32_t kOffBar = (kOffEpi + kEpiBytes + 7u) & ~7u;
  // full, empty, acc_full, acc_empty, drain
  static constexpr int kNumBars = 2 * kStages + 2 * kNumAcc + 1;
  static constexpr uint32_t kAHalfBytes = kATileBytes / 2;
  static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
  static constexpr uint32_t kSmemUsed = kOffAbort + 4;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;      // slack for aligning the base
  static constexpr uint32_t kIdesc = mma_idesc_f16(kBf16, kTileM, kBlockN, kBMnMajor);

  static_assert(kBlockN % 32 == 0 && kBlockN >= 32 && kBlockN <= 256, "MMA N");
  static_assert(kCtaGroup == 1 || kCtaGroup == 2, "cta group");
  static_assert(kStages >= 1 && kStages <= 32, "issued phases fit a 32-bit mask");
  static_assert(!kKPairs || (kCtaGroup == 1 && !kMulticastA && !kBMnMajor && !kTailSplit),
                "two k-blocks per stage: single-CTA K-major tiles, whole units of work");
  static_assert(kClusterPairs == 1 || (kClusterPairs == 2 && kCtaGroup == 2), "A multicast pairs CTA pairs");
  static_assert(kBRows % 8 == 0 && kBRows <= 256, "TMA box rows");
  static_assert(!kBMnMajor || kBRows % 64 == 0, "MN-major B is loaded in 64-wide boxes");
  static_assert(kATileBytes % 1024 == 0 && kBTileBytes % 1024 == 0, "swizzle atoms stay 1024-aligned");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns");
  static_assert(kOffBar >= kOffEpi + kEpiBytes, "barriers after every buffer");
  static_assert(kOffEpi % 1024 == 0, "TMA-store staging boxes stay swizzle-aligned");
  static_assert(kSmemBytes <= 232448, "fits the opt-in shared memory of one CTA");
};

// Tile index -> (tile row, tile column), grouped so that consecutive indices
// sweep `group_m` tile rows before moving to the next column; the last group
// may hold fewer rows.
__device__ __forceinline__ void tile_coords(const GemmArgs& a, int tile, int& tm, int& tn) {
  const int g = a.div_group.div(tile);
  const int first_m = g * a.group_m;
  const int in_group = tile - g * a.group_m * a.num_n_tiles;
  const bool full = first_m + a.group_m <= a.num_m_tiles;
  const int rows = full ? a.group_m : a.num_m_tiles - first_m;
  const int col = (full ? a.div_rows : a.div_last_rows).div(in_group);
  tm = first_m + (in_group - col * rows);
  tn = col;
}

// ---------------------------------------------------------------- work split

struct WorkItem {
  int tile;        // tile index in raster order
  int kb_begin;    // first k-block of this item
  int kb_end;      // one past the last k-block
  int sub;         // sub-tile index along N within a cut tile (0 when whole)
  int nsub;        // number of sub-tiles the tile is cut into (1 when whole)
  int nsub_log2;   // log2(nsub)
};

// First stream-K iteration of `worker`'s range.
__device__ __forceinline__ int64_t sk_range_begin(const GemmArgs& a, int worker) {
  return a.sk_iters * worker / a.sk_workers;
}

// Worker whose stream-K range holds iteration i (ranges are non-empty).
__device__ __forceinline__ int sk_worker_of(const GemmArgs& a, int64_t i) {
  int w = static_cast<int>(i * a.sk_workers / a.sk_iters);
  while (w + 1 < a.sk_workers && sk_range_begin(a, w + 1) <= i) ++w;
  while (w > 0 && sk_range_begin(a, w) > i) --w;
  return w;
}

// The sequence of work items of one worker: its stream-K range first, cut at
// tile boundaries (a contributed tail, whole tiles, then the head of the tile
// it finishes), then its whole tiles. Running the range first means every
// contributor's partial is written early, and the finisher's fix-up epilogue
// overlaps the main loop of the whole tiles that follow. Every role of a CTA
// walks the same sequence.
template <bool kTailSplit>
struct WorkCursor {
  int dp_next;
  int64_t sk_cur, sk_end;

  __device__ __forceinline__ WorkCursor(const GemmArgs& a, int worker)
      : dp_next(worker), sk_cur(0), sk_end(0) {
    if (a.sk_iters > 0 && worker < a.sk_workers) {
      sk_cur = sk_range_begin(a, worker);
      sk_end = sk_range_begin(a, worker + 1);
    }
  }

  __device__ __forceinline__ bool next(const GemmArgs& a, WorkItem& w) {
    if (sk_cur < sk_end) {
      const int64_t t = sk_cur / a.num_k_blocks;
      const int kb0 = static_cast<int>(sk_cur - t * a.num_k_blocks);
      const int64_t left = sk_end - sk_cur;
      const int kb1 = left < a.num_k_blocks - kb0 ? kb0 + static_cast<int>(left) : a.num_k_blocks;
      w.tile = a.dp_tiles + static_cast<int>(t);
      w.kb_begin = kb0;
      w.kb_end = kb1;
      w.sub = 0;
      w.nsub = 1;
      w.nsub_log2 = 0;
      sk_cur += kb1 - kb0;
      return true;
    }
    // whole tiles, then the sub-tiles of the cut tail tiles, round-robin
    // (32-bit arithmetic and shifts: the split is a power of two)
    if (dp_next < (kTailSplit ? a.dp_units : a.dp_tiles)) {
      if (!kTailSplit || dp_next < a.split_begin) {
        w.tile = dp_next;
        w.sub = 0;
        w.nsub = 1;
        w.nsub_log2 = 0;
      } else {
        const int u = dp_next - a.split_begin;
        w.tile = a.split_begin + (u >> a.split_log2);
        w.sub = u & (a.split - 1);
        w.nsub = a.split;
        w.nsub_log2 = a.split_log2;
      }
      w.kb_begin = 0;
      w.kb_end = a.num_k_blocks;
      dp_next += a.num_workers;
      return true;
    }
    return false;
  }
};

// First k-block of a rotated K walk for tile column `tile_col` (0 when the
// item does not cover all of K or rotation is off). Tile columns are spread
// over K by Fibonacci hashing (the fractional part of tile_col x 0.618...),
// so the tiles streaming their rows of B at the same time read different K
// offsets: rows of B lie a whole row pitch apart, and when every tile reads
// the same offset the concurrent reads fall on few DRAM banks. Tiles of one
// column (which share rows of B) start at the same k-block. The producer
// loads k-block rotate_kb(i) as the i-th of the item and the MMA consumes the
// ring in order, so C is the same sum up to the order of fp32 additions.
__device__ __forceinline__ int k_start(const GemmArgs& a, const WorkItem& w, int tile_col) {
  if (a.k_rotate == 0 || w.kb_begin != 0 || w.kb_end != a.num_k_blocks) return 0;
  const uint32_t h = static_cast<uint32_t>(tile_col) * 0x9E3779B9u;
  return static_cast<int>((static_cast<uint64_t>(h) * static_cast<uint32_t>(a.num_k_blocks)) >> 32);
}

__device__ __forceinline__ int rotate_kb(int kb, int start, int num_k_blocks) {
  const int r = kb + start;
  return r >= num_k_blocks ? r - num_k_blocks : r;
}

__device__ __forceinline__ uint64_t ld_acquire_gpu(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

// The last phase the producer issued into each stage of its ring (up to 32
// stages), held in two registers: a dynamically indexed array would live in
// local memory, and with this none of the kernels needs a stack frame.
struct IssuedPhases {
  uint32_t issued = 0u;   // bit s: some phase was issued into stage s
  uint32_t parity = 0u;   // bit s: the parity of that phase
  __device__ __forceinline__ void record(int s, uint32_t phase) {
    issued |= 1u << s;
    parity = (parity & ~(1u << s)) | ((phase & 1u) << s);
  }
  __device__ __forceinline__ bool any(int s) const { return ((issued >> s) & 1u) != 0u; }
  __device__ __forceinline__ uint32_t phase(int s) const { return (parity >> s) & 1u; }
};

template <class Cfg>
__device__ __forceinline__ void store_pair_bits(uint32_t& out, uint32_t lo, uint32_t hi) {
  const float flo = __uint_as_float(lo), fhi = __uint_as_float(hi);
  if constexpr (Cfg::kBf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(flo, fhi);
    out = *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(flo, fhi);
    out = *reinterpret_cast<uint32_t*>(&v);
  }
}

template <class Cfg>
struct Watchdog {
  const GemmArgs* args;
  volatile uint32_t* abort_flag;
  uint32_t abort_addr;   // shared address of the abort flag (for the peer CTA)

  // Wait for the phase of `bar` with parity `parity`; false on timeout or
  // when another role has already given up.
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    constexpr bool kCluster = Cfg::kClusterSize > 1;
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
    const uint64_t deadline = globaltimer_ns() + args->timeout_ns;
    while (true) {
      if (mbar_try_wait<kCluster>(bar, parity)) return true;
      if (*abort_flag) return false;
      if (globaltimer_ns() > deadline) {
        fail();
        return false;
      }
    }
  }

  // Wait until a global flag written by another CTA holds this launch's
  // epoch; false on timeout or when another role has already given up.
  __device__ __forceinline__ bool wait_flag(const uint64_t* flag) const {
    const uint64_t want = args->flag_epoch;
    if (ld_acquire_gpu(flag) == want) return true;
    const uint64_t deadline = globaltimer_ns() + args->timeout_ns;
    while (true) {
      if (ld_acquire_gpu(flag) == want) return true;
      if (*abort_flag) return false;
      if (globaltimer_ns() > deadline) {
        fail();
        return false;
      }
    }
  }

  // Bounded wait used while draining after a failure: never sets the flag.
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
    constexpr bool kCluster = Cfg::kClusterSize > 1;
    const uint64_t deadline = globaltimer_ns() + args->timeout_ns;
    while (!mbar_try_wait<kCluster>(bar, parity)) {
      if (globaltimer_ns() > deadline) return false;
    }
    return true;
  }

  __device__ __forceinline__ void fail() const {
    if (args->status != nullptr) atomicCAS(args->status, 0, kStatusTimeout);
    *abort_flag = 1u;
    if constexpr (Cfg::kClusterSize > 1) {
      const uint32_t me = cluster_ctarank();
      for (uint32_t r = 0; r < static_cast<uint32_t>(Cfg::kClusterSize); ++r)
        if (r != me) st_cluster_u32(map_to_cta(abort_addr, r), 1u);
    }
  }
};

template <class Cfg>
__global__ void __launch_bounds__(kNumThreads, 1) gemm_tn_sm103_kernel(const __grid_constant__ GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t base = smem_addr(smem);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t cluster_rank = (Cfg::kClusterSize > 1) ? cluster_ctarank() : 0u;
  const uint32_t cta_rank = (Cfg::kCtaGroup == 2) ? (cluster_rank & 1u) : 0u;   // position in the CTA pair
  const uint32_t pair = Cfg::kMulticastA ? (cluster_rank >> 1) : 0u;            // pair within the cluster
  const uint32_t pair_leader = cluster_rank & ~1u;
  const bool leader = cta_rank == 0;

  auto a_tile = [&](int s) { return base + Cfg::kOffA + s * Cfg::kStageA; };
  auto b_tile = [&](int s) { return base + Cfg::kOffB + s * Cfg::kStageB; };
  auto full_bar = [&](int s) { return base + Cfg::kOffBar + 8u * s; };
  auto empty_bar = [&](int s) { return base + Cfg::kOffBar + 8u * (Cfg::kStages + s); };
  auto acc_full_bar = [&](int a) { return base + Cfg::kOffBar + 8u * (2 * Cfg::kStages + a); };
  auto acc_empty_bar = [&](int a) { return base + Cfg::kOffBar + 8u * (2 * Cfg::kStages + Cfg::kNumAcc + a); };
  const uint32_t drain_bar = base + Cfg::kOffBar + 8u * (2 * Cfg::kStages + 2 * Cfg::kNumAcc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmemSlot);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffAbort);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      // full: the pair leader's expect-tx arrival and both CTAs' bytes
      mbar_init(full_bar(s), 1);
      // empty: one MMA commit per CTA pair that reads the stage
      mbar_init(empty_bar(s), Cfg::kClusterPairs);
    }
    for (int a = 0; a < Cfg::kNumAcc; ++a) {
      mbar_init(acc_full_bar(a), 1);
      mbar_init(acc_empty_bar(a), Cfg::kCtaGroup * kNumEpilogueWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_descriptor(&args.tmap_a);
    tma_prefetch_descriptor(&args.tmap_b);
  }
  if (warp == kMmaWarp) {
    tmem_alloc<Cfg::kCtaGroup>(smem_addr(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish<Cfg::kCtaGroup>();
  }
  tc_fence_before_sync();
  if constexpr (Cfg::kClusterSize > 1) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // The set-up above (barriers, TMEM, descriptor prefetch) may overlap the
  // end of the previous kernel in the stream; global memory is touched only
  // once that kernel has completed. Every thread but the producer waits for
  // it here. The producer first works out its first unit of work, which
  // depends on the launch's parameters alone, and waits just before its
  // first copy, so that this arithmetic may overlap the previous kernel too.
  // The next kernel may then be scheduled: it takes an SM only when a CTA of
  // this grid leaves it, and this grid is resident as a whole, so nothing
  // here waits on it.
  const bool producer_thread = warp == kProducerWarp && lane == 0;
  if (!producer_thread) {
    griddep_wait();
    griddep_launch_dependents();
  }

  const Watchdog<Cfg> wd{&args, abort_flag, smem_addr(const_cast<uint32_t*>(abort_flag))};
  const int worker = static_cast<int>(blockIdx.x) / Cfg::kClusterSize;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      const uint64_t pol_b = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      IssuedPhases issued;
      bool ok = true;
      bool dep_waited = false;   // griddep_wait() has returned
      int item_index = 0;
      WorkCursor<Cfg::kTailSplit> cursor(args, worker);
      WorkItem item;
      while (ok && cursor.next(args, item)) {
        int tm, tj;
        tile_coords(args, item.tile, tm, tj);
        const int tn = tj * Cfg::kClusterPairs + static_cast<int>(pair);
        const int a_row = tm * Cfg::kTileM + static_cast<int>(cta_rank) * Cfg::kBlockM;
        const int sub_n = Cfg::kBlockN >> item.nsub_log2;   // columns of this unit of work
        const int b_row = tn * Cfg::kBlockN + item.sub * sub_n + static_cast<int>(cta_rank) * (Cfg::kBRows >> item.nsub_log2);
        const void* tmap_b = item.nsub > 1 && !Cfg::kBMnMajor ? static_cast<const void*>(&args.tmap_b_split)
                                                              : static_cast<const void*>(&args.tmap_b);
        const uint32_t b_bytes = Cfg::kBTileBytes >> item.nsub_log2;
        // B of one k-block into this CTA's stage buffer, completing on `bar`
        // (the pair leader's barrier for CTA pairs): one box [rows x 64 K]
        // when K-major, or 64-wide N boxes of [64 K x 64 N] when MN-major.
        auto load_b = [&](int stage_, uint32_t bar, int kb_) {
          if constexpr (Cfg::kBMnMajor) {
            const int boxes = (Cfg::kBRows >> item.nsub_log2) / 64;
            for (int j = 0; j < boxes; ++j) {
              if constexpr (Cfg::kCtaGroup == 2) {
                tma_load_2d_pair(tmap_b, b_tile(stage_) + j * Cfg::kBMnBoxBytes, bar, b_row + 64 * j,
                                 kb_ * Cfg::kBlockK);
              } else {
                tma_load_2d(tmap_b, b_tile(stage_) + j * Cfg::kBMnBoxBytes, bar, b_row + 64 * j, kb_ * Cfg::kBlockK);
              }
            }
          } else if constexpr (Cfg::kCtaGroup == 2) {
            tma_load_2d_pair(tmap_b, b_tile(stage_), bar, kb_ * Cfg::kBlockK, b_row);
          } else if constexpr (Cfg::kKPairs) {
            tma_load_3d(tmap_b, b_tile(stage_), bar, 0, b_row, 2 * kb_);   // k-blocks 2 kb_, 2 kb_ + 1
          } else if (args.b_evict_first) {
            tma_load_2d_hint(tmap_b, b_tile(stage_), bar, kb_ * Cfg::kBlockK, b_row, pol_b);
          } else {
            tma_load_2d(tmap_b, b_tile(stage_), bar, kb_ * Cfg::kBlockK, b_row);
          }
        };
        const int kstart = k_start(args, item, tj);
        // stages of this unit of work (kKb k-blocks each; with two, every
        // unit covers all of K from k-block 0)
        const int st_begin = item.kb_begin / Cfg::kKb;
        const int st_end = (item.kb_end + Cfg::kKb - 1) / Cfg::kKb;
        for (int kb_i = st_begin; kb_i < st_end; ++kb_i) {
          if (!wd.wait(empty_bar(stage), phase ^ 1u)) {
            ok = false;
            break;
          }
          if (!dep_waited) {
            griddep_wait();
            griddep_launch_dependents();
            dep_waited = true;
          }
          const int kb = rotate_kb(kb_i, kstart, args.num_k_blocks);
          const uint32_t fb = full_bar(stage);
          const bool drop = item_index == 0 && kb_i == args.drop_load_kb;
          if constexpr (Cfg::kMulticastA) {
            // A: this CTA loads one 64-row half of its A block and multicasts
            // it to the CTA at the same position in the other pair; every
            // destination pair's leader counts the bytes, so the leader
            // expects both halves for both of its CTAs plus both B tiles,
            // the same total as without multicast.
            if (leader) mbar_arrive_expect_tx(fb, Cfg::kCtaGroup * (Cfg::kATileBytes + b_bytes));
            if (!drop) {
              const int x = kb * Cfg::kBlockK;
              const uint16_t mask = static_cast<uint16_t>((1u << cta_rank) | (1u << (2u + cta_rank)));
              tma_load_2d_multicast_pair(&args.tmap_a, a_tile(stage) + pair * Cfg::kAHalfBytes, fb & 0xFEFFFFFFu, x,
                                         a_row + static_cast<int>(pair) * (Cfg::kBlockM / 2), mask);
              load_b(stage, map_to_cta(fb, pair_leader), kb);
            }
            issued.record(stage, phase);
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (leader) mbar_arrive_expect_tx(fb, Cfg::kCtaGroup * Cfg::kKb * (Cfg::kATileBytes + b_bytes));
          if (!drop) {
            const int x = kb * Cfg::kBlockK;
            if constexpr (Cfg::kCtaGroup == 2) {
              const uint32_t fb_leader = map_to_cta(fb, pair_leader);
              tma_load_2d_pair(&args.tmap_a, a_tile(stage), fb_leader, x, a_row);
              load_b(stage, fb_leader, kb);
            } else if constexpr (Cfg::kKPairs) {
              tma_load_3d(&args.tmap_a, a_tile(stage), fb, 0, a_row, 2 * kb);   // k-blocks 2 kb, 2 kb + 1
              load_b(stage, fb, kb);
            } else {
              tma_load_2d(&args.tmap_a, a_tile(stage), fb, x, a_row);
              load_b(stage, fb, kb);
            }
          }
          issued.record(stage, phase);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        ++item_index;
      }
      if (!dep_waited) {
        griddep_wait();
        griddep_launch_dependents();
      }
      // Loads may still be landing if another role gave up: wait (bounded)
      // for the last phase issued into every stage before the CTA may exit.
      // On the normal path these phases have completed already. The
      // leader's full barriers count the peer's bytes (and, with multicast,
      // the other pair's halves) too.
      for (int s = 0; s < Cfg::kStages; ++s) {
        if (issued.any(s) && leader) wd.drain(full_bar(s), issued.phase(s));
      }
    }
  } else if (warp == kMmaWarp) {
    if (leader && lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      WorkCursor<Cfg::kTailSplit> cursor(args, worker);
      WorkItem item;
      while (ok && cursor.next(args, item)) {
        if (!wd.wait(acc_empty_bar(acc), acc_phase ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::kAccCols);
        // a sub-tile of a cut tile multiplies with N = block_n / nsub
        const uint32_t idesc =
            item.nsub == 1 ? Cfg::kIdesc
                           : mma_idesc_f16(Cfg::kBf16, Cfg::kTileM, Cfg::kBlockN >> item.nsub_log2, Cfg::kBMnMajor);
        const int st_begin = item.kb_begin / Cfg::kKb;
        const int st_end = (item.kb_end + Cfg::kKb - 1) / Cfg::kKb;
        for (int kb = st_begin; kb < st_end; ++kb) {
          if (!wd.wait(full_bar(stage), phase)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // one K=16 step: 32 bytes along a K-major row, or two 1024-byte
          // 8-row K groups of an MN-major tile
          constexpr uint32_t kBStep = Cfg::kBMnMajor ? (2048u >> 4) : 2u;
          constexpr int kSteps = Cfg::kBlockK / Cfg::kMmaK;   // per k-block
#pragma unroll
          for (int kb2 = 0; kb2 < Cfg::kKb; ++kb2) {   // k-blocks of the stage
            const uint64_t a_desc = sw128_kmajor_desc(a_tile(stage) + kb2 * Cfg::kATileBytes);
            const uint64_t b_desc = Cfg::kBMnMajor
                                        ? sw128_mnmajor_desc(b_tile(stage), Cfg::kBMnBoxBytes)
                                        : sw128_kmajor_desc(b_tile(stage) + kb2 * Cfg::kBTileBytes);
#pragma unroll
            for (int kk = 0; kk < kSteps; ++kk) {
              // advancing 16 elements along K = 32 bytes = 2 descriptor units
              mma_f16<Cfg::kCtaGroup>(d_tmem, a_desc + 2u * kk, b_desc + kBStep * kk, idesc,
                                      (kb > st_begin || kb2 > 0 || kk > 0) ? 1u : 0u);
            }
          }
          if constexpr (Cfg::kMulticastA) {
            mma_commit_pair(empty_bar(stage), 0xF);   // both pairs' buffers hold halves of this A
          } else if constexpr (Cfg::kCtaGroup == 2) {
            mma_commit_pair(empty_bar(stage), 0x3);
          } else {
            mma_commit(empty_bar(stage));
          }
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (Cfg::kCtaGroup == 2) {
          mma_commit_pair(acc_full_bar(acc), static_cast<uint16_t>(0x3u << pair_leader));
        } else {
          mma_commit(acc_full_bar(acc));
        }
        if (++acc == Cfg::kNumAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs issued by this thread must finish before TMEM is freed.
      if constexpr (Cfg::kCtaGroup == 2) {
        mma_commit_pair(drain_bar, static_cast<uint16_t>(1u << cluster_rank));
      } else {
        mma_commit(drain_bar);
      }
      wd.drain(drain_bar, 0);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const uint32_t quarter = warp & 3u;           // TMEM lanes this warp may read
    const uint32_t epi_warp = warp - kFirstEpilogueWarp;
    const int half = static_cast<int>(epi_warp >> 2);   // this warp takes chunks half, half + 2, ...
    uint8_t* warp_stage = smem + Cfg::kOffEpi + epi_warp * Cfg::kEpiWarpBytes;
    uint32_t* stg = reinterpret_cast<uint32_t*>(warp_stage);
    const uint32_t stage_addr = smem_addr(warp_stage);
    const bool tma_store = args.c_tma_store != 0;
    int store_buf = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t acc_empty_leader0 =
        (Cfg::kCtaGroup == 2) ? map_to_cta(acc_empty_bar(0), pair_leader) : acc_empty_bar(0);
    uint16_t* cptr = static_cast<uint16_t*>(args.c);
    // fp32 partial rows of this thread: [chunk][128 rows][32] per CTA slot
    constexpr int kChunks = Cfg::kBlockN / 32;
    const int64_t row_in_cta = static_cast<int64_t>(quarter) * 32 + lane;
    bool ok = true;
    WorkCursor<Cfg::kTailSplit> cursor(args, worker);
    WorkItem item;
    while (ok && cursor.next(args, item)) {
      int tm, tj;
      tile_coords(args, item.tile, tm, tj);
      const int tn = tj * Cfg::kClusterPairs + static_cast<int>(pair);
      // warp-uniform outcome: the tcgen05 loads below are warp-collective
      if (!__all_sync(0xffffffffu, wd.wait(acc_full_bar(acc), acc_phase))) break;
      tc_fence_after_sync();
      const int row0 = tm * Cfg::kTileM + static_cast<int>(cta_rank) * Cfg::kBlockM + static_cast<int>(quarter) * 32;
      const int col_tile = tn * Cfg::kBlockN + item.sub * (Cfg::kBlockN >> item.nsub_log2);
      const uint32_t t_row = tmem_base + ((quarter * 32u) << 16) + static_cast<uint32_t>(acc * Cfg::kAccCols);
      // 32-column chunks of this tile that lie inside N (warp-uniform; 0 when
      // a multicast cluster's second pair lies wholly past N)
      const int chunks = max(0, min(kChunks >> item.nsub_log2, (args.n - col_tile + 31) / 32));
      if (chunks == 0) {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_leader0 + 8u * acc);
        if (++acc == Cfg::kNumAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
        continue;
      }
      // stream-K roles of this item: a contributor (does not hold the first
      // k-block) writes fp32 partial rows; the finisher (holds the first
      // k-block of a cut tile) adds the contributors' partials
      const bool contributor = item.kb_begin > 0;
      int first_contrib = 0, last_contrib = -1;
      if (!contributor && item.kb_end < args.num_k_blocks) {
        const int64_t t_local = item.tile - args.dp_tiles;
        first_contrib = worker + 1;
        last_contrib = sk_worker_of(args, (t_local + 1) * args.num_k_blocks - 1);
        for (int w = first_contrib; w <= last_contrib && ok; ++w) {
          const int cta = w * Cfg::kClusterSize + static_cast<int>(cluster_rank);
          ok = __all_sync(0xffffffffu, wd.wait_flag(args.flags + cta * kNumEpilogueWarps + epi_warp));
        }
        if (!ok) break;
      }
      // finisher: partial rows of the next chunk are loaded one chunk ahead
      const bool finisher = last_contrib >= first_contrib;
      // partial rows are stored as [cta][chunk][j][128 rows] float4s: the j-th
      // 16 bytes of every row of a chunk lie side by side, so each warp-wide
      // store or load of them moves 512 contiguous bytes
      auto partial_src = [&](int w, int chunk) {
        const int cta = w * Cfg::kClusterSize + static_cast<int>(cluster_rank);
        return reinterpret_cast<const float4*>(args.partials) +
               (static_cast<int64_t>(cta) * kChunks + chunk) * (8 * 128) + row_in_cta;
      };
      // this warp's last chunk (-1: none), after whose TMEM load it hands
      // the accumulator back to the MMA warp (every epilogue warp arrives once)
      const int my_last = chunks > half ? half + (((chunks - 1 - half) >> 1) << 1) : -1;
      auto hand_back = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if constexpr (Cfg::kCtaGroup == 2) {
            mbar_arrive_cluster(acc_empty_leader0 + 8u * acc);
          } else {
            mbar_arrive(acc_empty_bar(acc));
          }
        }
      };
      if (my_last < 0) hand_back();
      float4 pre[8];
      if (finisher && half < chunks) {
#pragma unroll
        for (int j = 0; j < 8; ++j) pre[j] = __ldcg(partial_src(first_contrib, half) + j * 128);
      }
      for (int chunk = half; chunk < chunks; chunk += 2) {
        const int col0 = col_tile + chunk * 32;
        uint32_t r[32];
        tmem_load_32x32(t_row + static_cast<uint32_t>(chunk * 32), r);
        tmem_load_wait();
        // the accumulator is in registers now: hand it back to the MMA warp
        if (chunk == my_last) hand_back();
        if (contributor) {
          float4* dst = reinterpret_cast<float4*>(args.partials) +
                        (static_cast<int64_t>(blockIdx.x) * kChunks + chunk) * (8 * 128) + row_in_cta;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j * 128] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          continue;
        }
        if (finisher) {
          // add the contributors' partials in worker order: the first one was
          // loaded ahead; the next chunk's first partial is issued now
          for (int w = first_contrib; w <= last_contrib; ++w) {
            float4 v[8];
            if (w == first_contrib) {
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] = pre[j];
              if (chunk + 2 < chunks) {
#pragma unroll
                for (int j = 0; j < 8; ++j) pre[j] = __ldcg(partial_src(first_contrib, chunk + 2) + j * 128);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] = __ldcg(partial_src(w, chunk) + j * 128);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + v[j].x);
              r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + v[j].y);
              r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + v[j].z);
              r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + v[j].w);
            }
          }
        }
        if constexpr (Cfg::kFused) {
          // fused epilogue on this thread's row (row0 + lane), columns
          // [col0, col0 + 32): scale, add the bias and beta * C, activate
          const int row = row0 + static_cast<int>(lane);
          const bool row_ok = row < args.m;
          const bool full = col0 + 32 <= args.n;
          const int64_t rbase = static_cast<int64_t>(row) * args.ldc + col0;
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = args.alpha * __uint_as_float(r[j]);
          if (args.bias != nullptr) {
            const float* bp = args.bias + col0;
            if (full && (reinterpret_cast<uintptr_t>(bp) & 15u) == 0) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 t = __ldg(reinterpret_cast<const float4*>(bp) + j);
                v[4 * j] += t.x;
                v[4 * j + 1] += t.y;
                v[4 * j + 2] += t.z;
                v[4 * j + 3] += t.w;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j < args.n) v[j] += __ldg(bp + j);
            }
          }
          if (args.beta != 0.0f && row_ok) {
            if (args.out_kind == 2) {
              // C's previous contents as e4m3 bytes, widened exactly
              const uint8_t* src = static_cast<const uint8_t*>(args.c) + rbase;
              if (full && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                  const uint4 t = reinterpret_cast<const uint4*>(src)[j];
                  const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    float f0, f1, f2, f3;
                    e4m3x2_to_f32(w4[q] & 0xFFFFu, f0, f1);
                    e4m3x2_to_f32(w4[q] >> 16, f2, f3);
                    v[16 * j + 4 * q] += args.beta * f0;
                    v[16 * j + 4 * q + 1] += args.beta * f1;
                    v[16 * j + 4 * q + 2] += args.beta * f2;
                    v[16 * j + 4 * q + 3] += args.beta * f3;
                  }
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  if (col0 + j < args.n) {
                    float f, unused;
                    e4m3x2_to_f32(src[j], f, unused);
                    v[j] += args.beta * f;
                  }
                }
              }
            } else if (args.out_kind == 1) {
              const float* src = static_cast<const float*>(args.c) + rbase;
              if (full && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float4 t = reinterpret_cast<const float4*>(src)[j];
                  v[4 * j] += args.beta * t.x;
                  v[4 * j + 1] += args.beta * t.y;
                  v[4 * j + 2] += args.beta * t.z;
                  v[4 * j + 3] += args.beta * t.w;
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (col0 + j < args.n) v[j] += args.beta * src[j];
              }
            } else {
              const uint16_t* src = static_cast<const uint16_t*>(args.c) + rbase;
              auto widen = [](uint32_t bits16) {
                if constexpr (Cfg::kBf16) {
                  return __uint_as_float(bits16 << 16);
                } else {
                  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
                }
              };
              if (full && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const uint4 t = reinterpret_cast<const uint4*>(src)[j];
                  const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    v[8 * j + 2 * q] += args.beta * widen(w4[q] & 0xFFFFu);
                    v[8 * j + 2 * q + 1] += args.beta * widen(w4[q] >> 16);
                  }
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (col0 + j < args.n) v[j] += args.beta * widen(src[j]);
              }
            }
          }
          if (args.activation == 1) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j], 0.0f);
          } else if (args.activation == 2) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
          if (args.out_kind == 2) {
            // e4m3 output: each row's 32 bytes go through the warp's staging
            // block (two 16-byte halves, swapped on every other group of four
            // rows so the writes spread over all banks), then each store
            // instruction writes the full 32 bytes of 16 rows
            uint32_t q8[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              q8[j] = cvt_e4m3x2(v[4 * j], v[4 * j + 1]) | (cvt_e4m3x2(v[4 * j + 2], v[4 * j + 3]) << 16);
            __syncwarp();
            const uint32_t flip = (lane >> 2) & 1u;
            st_shared_v4(stage_addr + lane * 32u + (flip * 16u), q8[0], q8[1], q8[2], q8[3]);
            st_shared_v4(stage_addr + lane * 32u + ((flip ^ 1u) * 16u), q8[4], q8[5], q8[6], q8[7]);
            __syncwarp();
            const uint32_t half16 = lane & 1u;
            const int col = col0 + static_cast<int>(half16) * 16;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const uint32_t rr = static_cast<uint32_t>(i) * 16u + (lane >> 1);
              const int row = row0 + static_cast<int>(rr);
              const uint4 val =
                  *reinterpret_cast<const uint4*>(warp_stage + rr * 32u + ((half16 ^ ((rr >> 2) & 1u)) * 16u));
              if (row >= args.m || col >= args.n) continue;
              uint8_t* dst = static_cast<uint8_t*>(args.c) + static_cast<int64_t>(row) * args.ldc + col;
              if (col + 16 <= args.n && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
                *reinterpret_cast<uint4*>(dst) = val;
              } else {
                const uint32_t w[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
                for (int q = 0; q < 16; ++q)
                  if (col + q < args.n) dst[q] = static_cast<uint8_t>(w[q >> 2] >> ((q & 3) * 8));
              }
            }
            continue;
          }
          if (args.out_kind == 1) {
            // fp32 output: the warp's 32 rows x 32 values go through its 4 KiB
            // staging block (16-byte units XOR-swizzled by row), then each
            // store instruction writes 128 contiguous bytes of four rows
            // instead of 16 bytes of 32 rows
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u)
              st_shared_v4(stage_addr + lane * 128u + ((static_cast<uint32_t>(u) ^ (lane & 7u)) * 16u),
                           __float_as_uint(v[4 * u]), __float_as_uint(v[4 * u + 1]), __float_as_uint(v[4 * u + 2]),
                           __float_as_uint(v[4 * u + 3]));
            __syncwarp();
            const uint32_t unit = lane & 7u;
            const int col = col0 + static_cast<int>(unit) * 4;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t rr = static_cast<uint32_t>(i) * 4u + (lane >> 3);
              const int row = row0 + static_cast<int>(rr);
              const float4 val = *reinterpret_cast<const float4*>(warp_stage + rr * 128u + ((unit ^ (rr & 7u)) * 16u));
              if (row >= args.m || col >= args.n) continue;
              float* dst = static_cast<float*>(args.c) + static_cast<int64_t>(row) * args.ldc + col;
              if (col + 4 <= args.n && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
                *reinterpret_cast<float4*>(dst) = val;
              } else {
                const float e[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  if (col + q < args.n) dst[q] = e[q];
              }
            }
            continue;
          }
        }
        // this thread holds row (row0 + lane), columns [col0, col0 + 32)
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) store_pair_bits<Cfg>(packed[j], r[2 * j], r[2 * j + 1]);
        // The TMA store writes whole 32 x 32 boxes: only boxes that lie inside
        // M and N go that way (a box crossing N is not clipped element by
        // element); edge chunks use the predicated element stores.
        const bool box_inside = col0 + 32 <= args.n && row0 + 32 <= args.m;
        if (tma_store && box_inside) {
          // the TMA store that last read this buffer must be done with it
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
          const uint32_t buf = stage_addr + static_cast<uint32_t>(store_buf) * 2048u;
          // 64-byte-swizzled 32 x 32 box: 16-byte chunk j of row r sits at
          // chunk position j ^ ((r >> 1) & 3) of the row's 64 bytes
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t pos = static_cast<uint32_t>(j) ^ ((lane >> 1) & 3u);
            st_shared_v4(buf + lane * 64u + pos * 16u, packed[4 * j], packed[4 * j + 1], packed[4 * j + 2],
                         packed[4 * j + 3]);
          }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&args.tmap_c, buf, col0, row0);
            bulk_commit_group();
          }
          store_buf ^= 1;
        } else {
          if (tma_store) {
            // the staging block doubles as the TMA boxes: let pending stores finish reading it
            if (lane == 0) bulk_wait_group_read<0>();
            __syncwarp();
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) stg[lane * Cfg::kStageRowWords + j] = packed[j];
          __syncwarp();
          // transpose through shared memory: each store instruction writes 32
          // consecutive columns of one row. All 32 values are read back
          // before the first store, and the row pointer steps by ldc, so the
          // stores issue back to back (with a load-store pair per row and a
          // 64-bit row offset each time, the last tile's epilogue of the
          // ragged workload took 7.7 us; this way 3.3 us)
          const int col = col0 + static_cast<int>(lane);
          uint16_t vals[32];
#pragma unroll
          for (int rr = 0; rr < 32; ++rr) vals[rr] = reinterpret_cast<const uint16_t*>(stg + rr * Cfg::kStageRowWords)[lane];
          if (col < args.n) {
            const int rows_here = min(32, args.m - row0);
            uint16_t* p = cptr + static_cast<int64_t>(row0) * args.ldc + col;
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
              if (rr < rows_here) *p = vals[rr];
              p += args.ldc;
            }
          }
          __syncwarp();
        }
      }
      if (contributor) {
        // publish this warp's partial rows: each lane's writes are made
        // visible at GPU scope before lane 0 raises the flag
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(args.flags + blockIdx.x * kNumEpilogueWarps + epi_warp, args.flag_epoch);
      }
      if (++acc == Cfg::kNumAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (tma_store && lane == 0) bulk_wait_group_all();   // stores complete before the CTA exits
    __syncwarp();
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before_sync();
  if constexpr (Cfg::kClusterSize > 1) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc<Cfg::kCtaGroup>(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace gemm_tn_dev
