// sm103_flash_attn.cu -- the attention forward pass on the GEMM's pipeline:
// O = softmax(scale * Q K^T, causal mask) V for Q, K, V, O of shape
// [batch, seq, heads, dim], dim 64 or 128, fp16 or bf16.
//
// "TileLang: a tile language one level below Triton", section "FlashAttention:
// online softmax as tile code": a CTA owns a block of queries and walks the
// keys tile by tile, keeping the row maximum and row sum of an online softmax;
// the accumulated output is rescaled when the maximum grows, and divided by
// the row sum once at the end. exp2 is used with log2(e) folded into the scale.
// The causal mask stops the walk after the diagonal tile and masks inside it.
//
// The sm_103a mapping: one CTA owns two 128-query tiles (t = 0, 1) of one
// (batch, head) and walks 128-key tiles j.
//   warp 0      TMA producer: Q_0 and Q_1 once, then K_j and V_j into rings
//               (64-element boxes, 128-byte swizzle; the 3-D tensor maps
//               {heads*dim, seq, batch} zero-fill rows past seq).
//   warp 1      MMA issuer (one thread). Per key tile and query tile:
//               O_t += P_t V_j (M = 128, N = dim, K = 128 keys; P read from
//               tensor memory, V through an MN-major shared-memory descriptor,
//               no transpose), then S_t = Q_t K_{j+1}^T (M = N = 128, K = dim)
//               into the same TMEM columns. Tensor memory holds S_0, S_1 (P_t
//               is written over the first half of S_t) and O_0, O_1.
//   warps 2-9   softmax, four warps per query tile: row r of tile t is TMEM
//               lane r and belongs to one thread. Per key tile the thread
//               loads the row's 128 scores, writes P = exp2(s * scale * log2e
//               - max), rounded to the input type, over them (two values per
//               column), rescales its O row when needed, and at the end
//               divides by the row sum and stores the row.
// The two query tiles alternate on the tensor cores: while the softmax warps
// of tile 0 work on S_0, the tensor cores run P_1 V and the next Q_1 K^T, and
// the other way round, so the exp2 work of one tile overlaps the products of
// the other. P never passes through shared memory, whose bandwidth the operand
// reads of the two products and the TMA writes of K and V already load.
//
// Grid order: work units walk the query-tile pairs of a group of heads whose
// K and V fit in L2 together, so the units of one head share K and V through
// L2; with the causal mask the heaviest units (the last query tiles, which
// walk the most keys) of a group start first.
//
// Differences from the section's loop: the reference maximum of a row is
// only moved when a tile's maximum exceeds it by more than 2^8 (then O and the
// row sum are rescaled); otherwise the probabilities are taken against the
// old maximum (values up to 2^8, exact in fp16 and bf16 range). The result is
// the same softmax -- the final division uses the same reference for the
// numerator and the row sum -- with far fewer O rescales. After the first key
// tile the probabilities are computed against the current reference at once;
// since none of them can exceed 2^8 unless their sum does, the tile's maximum
// is only taken when the row sum passes 2^8, and only a warp in which a row's
// maximum moved computes them again. That keeps the pass over the scores for
// their maximum off the path between the two products.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gemm_tn_internal.h"
#include "sm103_ptx.cuh"

namespace gemm_tn_dev {

namespace fa {

constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kBlockM = 128;       // queries per query tile (TMEM lanes)
constexpr int kBlockN = 128;       // keys per key tile
constexpr int kTiles = 2;          // query tiles per CTA
constexpr int kStatusTimeout = 6;  // == GEMM_TN_ERR_TIMEOUT
// log2 of the largest factor by which probabilities may exceed 1 before the
// row's reference maximum is moved
constexpr float kRescaleThreshold = 8.0f;

template <int kDim_, bool kBf16_>
struct Cfg {
  static constexpr int kDim = kDim_;
  static constexpr bool kBf16 = kBf16_;
  static constexpr int kNumThreads = 64 + 128 * kTiles;   // producer, MMA, 4 softmax warps per query tile
  // registers per thread for one CTA per SM: each of the four SM
  // sub-partitions holds 16384 registers and ceil(warps / 4) of the warps
  // (multiples of 8 per thread)
  static constexpr int kMaxRegs = (16384 / 32 / ((kNumThreads / 32 + 3) / 4)) / 8 * 8;
  static constexpr int kDimBoxes = kDim / 64;             // 64-element (128-byte) boxes across dim
  static constexpr uint32_t kBoxBytes = 128u * 128u;      // 128 rows x 128 bytes
  static constexpr uint32_t kTileBytes = kDimBoxes * kBoxBytes;
  // K and V ring depths: as deep as shared memory allows (K is needed first)
  static constexpr int kKStages = kDim == 64 ? 6 : 3;
  static constexpr int kVStages = kDim == 64 ? 4 : 2;
  static constexpr uint32_t kOffQ = 0;                    // Q_0, Q_1
  static constexpr uint32_t kOffK = kOffQ + kTiles * kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
  // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2], p_full[2], o_done[2], drain
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 3 * kTiles + 1;
  static constexpr uint32_t kOffTmemSlot = kOffBar + 8u * kNumBars;
  static constexpr uint32_t kOffAbort = kOffTmemSlot + 4u;
  static constexpr uint32_t kSmemBytes = kOffAbort + 4u + 1024u;   // + slack to align the base to 1024
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;      // S_t: 128 fp32 columns at 128 t (P_t over half of them)
  static constexpr uint32_t kColO = 256;    // O_t: dim fp32 columns at 256 + dim t
  static constexpr uint32_t kIdescS = mma_idesc_f16(kBf16, kBlockM, kBlockN, false);
  static constexpr uint32_t kIdescO = mma_idesc_f16(kBf16, kBlockM, kDim, true);
  static_assert(kDim == 64 || kDim == 128, "head dim 64 or 128");
  static_assert(kSmemBytes <= 227u * 1024u, "shared memory budget");
  static_assert(kColO + kTiles * kDim <= kTmemCols, "TMEM budget");
};

struct Watch {
  const FlashArgs* args;
  volatile uint32_t* abort_flag;

  // Wait for the phase of `bar` with parity `parity`; false on timeout or when
  // another role has given up.
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (mbar_try_wait<false, false>(bar, parity)) return true;
    const uint64_t deadline = globaltimer_ns() + args->timeout_ns;
    while (true) {
      if (mbar_try_wait<false, false>(bar, parity)) return true;
      if (*abort_flag) return false;
      if (globaltimer_ns() > deadline) {
        if (args->status != nullptr) atomicCAS(args->status, 0, kStatusTimeout);
        *abort_flag = 1u;
        return false;
      }
    }
  }

  // Bounded wait while draining after a failure; never raises the flag.
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
    const uint64_t deadline = globaltimer_ns() + args->timeout_ns;
    while (!mbar_try_wait<false, false>(bar, parity)) {
      if (globaltimer_ns() > deadline) return false;
    }
    return true;
  }
};

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t out;
  if constexpr (kBf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    out = *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    out = *reinterpret_cast<uint32_t*>(&v);
  }
  return out;
}

}  // namespace fa

template <class C>
__global__ void __launch_bounds__(C::kNumThreads) __maxnreg__(C::kMaxRegs)
    flash_attn_fwd_kernel(const __grid_constant__ FlashArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t base = smem_addr(smem);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  // work unit: groups of args.head_group (batch, head) pairs, query-tile
  // pairs of a group interleaved across its heads, heaviest first when causal
  const int n_units = args.num_q_tiles;   // 256-query units per head
  const int bh_count = args.batch * args.heads;
  const int group = static_cast<int>(blockIdx.x) / (args.head_group * n_units);
  const int first_bh = group * args.head_group;
  const int heads_here = min(args.head_group, bh_count - first_bh);
  const int rem = static_cast<int>(blockIdx.x) - group * args.head_group * n_units;
  const int unit_rank = rem / heads_here;
  const int bh = first_bh + rem % heads_here;
  const int unit = args.causal ? n_units - 1 - unit_rank : unit_rank;
  const int b = bh / args.heads;
  const int h = bh % args.heads;
  const int q0 = unit * fa::kTiles * fa::kBlockM;   // first query of tile 0
  // key tiles each query tile walks: through its diagonal when causal
  auto key_tiles = [&](int t) {
    const int end = args.causal ? min(args.seq, q0 + (t + 1) * fa::kBlockM) : args.seq;
    return (end + fa::kBlockN - 1) / fa::kBlockN;
  };
  const int n0 = key_tiles(0), n1 = key_tiles(1);   // n0 <= n1
  const int x0 = h * C::kDim;   // column of this head in the {heads*dim, seq, batch} maps

  auto q_tile = [&](int t) { return base + C::kOffQ + t * C::kTileBytes; };
  auto k_tile = [&](int s) { return base + C::kOffK + s * C::kTileBytes; };
  auto v_tile = [&](int s) { return base + C::kOffV + s * C::kTileBytes; };
  auto bar = [&](int i) { return base + C::kOffBar + 8u * i; };
  constexpr int kVBar = 1 + 2 * C::kKStages;      // first V barrier
  constexpr int kTBar = kVBar + 2 * C::kVStages;  // first per-query-tile barrier
  const uint32_t q_full = bar(0);
  auto k_full = [&](int s) { return bar(1 + s); };
  auto k_empty = [&](int s) { return bar(1 + C::kKStages + s); };
  auto v_full = [&](int s) { return bar(kVBar + s); };
  auto v_empty = [&](int s) { return bar(kVBar + C::kVStages + s); };
  auto s_full = [&](int t) { return bar(kTBar + t); };
  auto p_full = [&](int t) { return bar(kTBar + fa::kTiles + t); };
  auto o_done = [&](int t) { return bar(kTBar + 2 * fa::kTiles + t); };
  const uint32_t drain_bar = bar(kTBar + 3 * fa::kTiles);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffAbort);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int t = 0; t < fa::kTiles; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), 4);   // one arrival per softmax warp of the tile
      mbar_init(o_done(t), 1);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == fa::kProducerWarp && lane == 0) {
    tma_prefetch_descriptor(&args.tmap_q);
    tma_prefetch_descriptor(&args.tmap_k);
    tma_prefetch_descriptor(&args.tmap_v);
  }
  if (warp == fa::kMmaWarp) {
    tmem_alloc<1>(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish<1>();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // The set-up above may overlap the end of the previous kernel in the
  // stream; global memory is touched only once that kernel has completed.
  // The next kernel is scheduled only after every CTA of this grid has run
  // this trigger (so after the last one has started), so it never holds an
  // SM that a CTA of this grid still waits for.
  griddep_wait();
  griddep_launch_dependents();
  const fa::Watch wd{&args, abort_flag};

  if (warp == fa::kProducerWarp) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int issued_k[C::kKStages], issued_v[C::kVStages];
      for (int s = 0; s < C::kKStages; ++s) issued_k[s] = -1;
      for (int s = 0; s < C::kVStages; ++s) issued_v[s] = -1;
      mbar_arrive_expect_tx(q_full, fa::kTiles * C::kTileBytes);
      for (int t = 0; t < fa::kTiles; ++t)
        for (int c = 0; c < C::kDimBoxes; ++c)
          tma_load_3d(&args.tmap_q, q_tile(t) + c * C::kBoxBytes, q_full, x0 + 64 * c, q0 + t * fa::kBlockM, b);
      const bool drop_here = blockIdx.x == 0;
      for (int j = 0; j < n1; ++j) {
        const int s = j % C::kKStages;
        const uint32_t ph = static_cast<uint32_t>(j / C::kKStages) & 1u;
        if (!wd.wait(k_empty(s), ph ^ 1u)) break;
        mbar_arrive_expect_tx(k_full(s), C::kTileBytes);
        if (!(drop_here && j == args.drop_load_block)) {
          for (int c = 0; c < C::kDimBoxes; ++c)
            tma_load_3d(&args.tmap_k, k_tile(s) + c * C::kBoxBytes, k_full(s), x0 + 64 * c, j * fa::kBlockN, b);
        }
        issued_k[s] = static_cast<int>(ph);
        const int sv = j % C::kVStages;
        const uint32_t phv = static_cast<uint32_t>(j / C::kVStages) & 1u;
        if (!wd.wait(v_empty(sv), phv ^ 1u)) break;
        mbar_arrive_expect_tx(v_full(sv), C::kTileBytes);
        for (int c = 0; c < C::kDimBoxes; ++c)
          tma_load_3d(&args.tmap_v, v_tile(sv) + c * C::kBoxBytes, v_full(sv), x0 + 64 * c, j * fa::kBlockN, b);
        issued_v[sv] = static_cast<int>(phv);
      }
      // Loads may still be landing if another role gave up: wait (bounded)
      // for every phase issued before the CTA may exit.
      wd.drain(q_full, 0);
      for (int s = 0; s < C::kKStages; ++s)
        if (issued_k[s] >= 0) wd.drain(k_full(s), static_cast<uint32_t>(issued_k[s]));
      for (int s = 0; s < C::kVStages; ++s)
        if (issued_v[s] >= 0) wd.drain(v_full(s), static_cast<uint32_t>(issued_v[s]));
    }
  } else if (warp == fa::kMmaWarp) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      // S_t = Q_t K_j^T into TMEM columns 128 t
      auto issue_s = [&](int t, int j) {
        const int s = j % C::kKStages;
        const uint32_t t_s = tmem_base + C::kColS + 128u * static_cast<uint32_t>(t);
#pragma unroll
        for (int c = 0; c < C::kDimBoxes; ++c) {
          const uint64_t a_desc = sw128_kmajor_desc(q_tile(t) + c * C::kBoxBytes);
          const uint64_t b_desc = sw128_kmajor_desc(k_tile(s) + c * C::kBoxBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // 16 elements of dim = 32 bytes = 2 descriptor units
            mma_f16<1>(t_s, a_desc + 2u * kk, b_desc + 2u * kk, C::kIdescS, (c | kk) != 0 ? 1u : 0u);
        }
        mma_commit(s_full(t));
      };
      // O_t += P_t V_j; P_t of keys 64 h .. 64 h + 63 lies over the first 32
      // columns of the 64 score columns of those keys
      auto issue_pv = [&](int t, int j) {
        const int s = j % C::kVStages;
        const uint64_t v_desc = sw128_mnmajor_desc(v_tile(s), C::kBoxBytes);
        const uint32_t t_p = tmem_base + C::kColS + 128u * static_cast<uint32_t>(t);
        const uint32_t t_o = tmem_base + C::kColO + static_cast<uint32_t>(C::kDim * t);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // 16 keys: 8 columns of P; 16 rows of 128 bytes of V
          mma_f16_tmem_a(t_o, t_p + 64u * static_cast<uint32_t>(kk >> 2) + 8u * static_cast<uint32_t>(kk & 3), v_desc + ((static_cast<uint32_t>(kk) * 2048u) >> 4), C::kIdescO,
                         (j > 0 || kk > 0) ? 1u : 0u);
      };
      auto wait_k = [&](int j) {
        return wd.wait(k_full(j % C::kKStages), static_cast<uint32_t>(j / C::kKStages) & 1u);
      };
      bool ok = wd.wait(q_full, 0) && wait_k(0);
      if (ok) {
        tc_fence_after_sync();
        issue_s(0, 0);
        issue_s(1, 0);
        mma_commit(k_empty(0));
      }
      for (int j = 0; ok && j < n1; ++j) {
        if (!wd.wait(v_full(j % C::kVStages), static_cast<uint32_t>(j / C::kVStages) & 1u)) {
          ok = false;
          break;
        }
        bool k_ready = false;   // K_{j+1} waited for
        for (int t = 0; t < fa::kTiles; ++t) {
          if (t == 0 && j >= n0) continue;   // tile 0 ends at its diagonal key tile
          if (!wd.wait(p_full(t), static_cast<uint32_t>(j) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_pv(t, j);
          if (t == fa::kTiles - 1) mma_commit(v_empty(j % C::kVStages));
          const bool t_next = j + 1 < (t == 0 ? n0 : n1);   // this tile walks key tile j + 1
          if (t_next) {
            if (!k_ready) {
              if (!wait_k(j + 1)) {
                ok = false;
                break;
              }
              k_ready = true;
              tc_fence_after_sync();
            }
            issue_s(t, j + 1);
            if (t == fa::kTiles - 1) mma_commit(k_empty((j + 1) % C::kKStages));
          } else {
            mma_commit(o_done(t));
          }
        }
      }
      // every MMA issued here must finish before TMEM is freed
      mma_commit(drain_bar);
      wd.drain(drain_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int t = (static_cast<int>(warp) - fa::kFirstSoftmaxWarp) >> 2;   // query tile
    const uint32_t quarter = warp & 3u;                                    // TMEM lanes 32*quarter ..
    const int r = static_cast<int>(quarter * 32u + lane);                  // row of the tile
    const int q_row = q0 + t * fa::kBlockM + r;
    const int n_t = t == 0 ? n0 : n1;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const uint32_t t_s = tmem_base + lane_off + C::kColS + 128u * static_cast<uint32_t>(t);
    // P of keys k lies at column 64 (k / 64) + (k % 64) / 2 of S_t, over scores
    // this thread has already read
    auto p_col = [&](int key) { return t_s + static_cast<uint32_t>(64 * (key / 64) + (key % 64) / 2); };
    const uint32_t t_o = tmem_base + lane_off + C::kColO + static_cast<uint32_t>(C::kDim * t);
    const float c_log2 = args.scale_log2;
    // keys this row may see: k < limit
    const int limit = args.causal ? min(q_row + 1, args.seq) : args.seq;
    // waits with a warp-uniform outcome: the tcgen05 loads and stores that
    // follow them are warp-collective
    auto warp_wait = [&](uint32_t bar_addr, uint32_t parity) {
      return __all_sync(0xffffffffu, wd.wait(bar_addr, parity));
    };
    float m_ref = -INFINITY;   // reference maximum, in units of scale * log2e
    float l = 0.0f;            // row sum of probabilities, against m_ref
    bool ok = true;
    for (int j = 0; j < n_t && ok; ++j) {
      // S_t for key tile j is complete, and with it P_t V_{j-1}: O_t is stable
      if (!warp_wait(s_full(t), static_cast<uint32_t>(j) & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      float sv[128];
      {
        uint32_t raw[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_load_32x32(t_s + 32u * c, raw[c]);
        tmem_load_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[c * 32 + e] = __uint_as_float(raw[c][e]);
      }
      const int key0 = j * fa::kBlockN;
      if (key0 + fa::kBlockN > limit) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (key0 + e >= limit) sv[e] = -INFINITY;
      }
      // probabilities against neg_m into the P columns; returns their sum
      // The scaling and the four running sums use packed fp32 pairs (one
      // instruction for two values, the same fp32 arithmetic per value): the
      // pass is bound by issue slots as much as by the exponential unit.
      auto exp_pass = [&](float neg_m) {
        const uint64_t cc = f32x2_pack(c_log2, c_log2), mm = f32x2_pack(neg_m, neg_m);
        uint64_t s01 = f32x2_pack(0.0f, 0.0f), s23 = f32x2_pack(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];   // 32 scores -> 16 columns of P
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float* x = sv + 32 * c + e;
            float a0, a1, a2, a3;
            f32x2_unpack(f32x2_fma(f32x2_pack(x[0], x[1]), cc, mm), a0, a1);
            f32x2_unpack(f32x2_fma(f32x2_pack(x[2], x[3]), cc, mm), a2, a3);
            const float p0 = ex2_approx(a0);
            const float p1 = ex2_approx(a1);
            const float p2 = ex2_approx(a2);
            const float p3 = ex2_approx(a3);
            s01 = f32x2_add(s01, f32x2_pack(p0, p1));
            s23 = f32x2_add(s23, f32x2_pack(p2, p3));
            pk[e / 2] = fa::pack2<C::kBf16>(p0, p1);
            pk[e / 2 + 1] = fa::pack2<C::kBf16>(p2, p3);
          }
          tmem_store_32x16(p_col(32 * c), pk);
        }
        float sum0, sum1, sum2, sum3;
        f32x2_unpack(s01, sum0, sum1);
        f32x2_unpack(s23, sum2, sum3);
        return (sum0 + sum1) + (sum2 + sum3);
      };
      auto row_max = [&]() {
        float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
        for (int e = 4; e < 128; e += 4) {
          mx0 = fmaxf(mx0, sv[e]);
          mx1 = fmaxf(mx1, sv[e + 1]);
          mx2 = fmaxf(mx2, sv[e + 2]);
          mx3 = fmaxf(mx3, sv[e + 3]);
        }
        return fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      };
      float alpha = 1.0f;
      float sum;
      if (j == 0) {
        // first tile: the reference maximum is the tile's maximum
        m_ref = row_max() * c_log2;
        sum = exp_pass(-m_ref);
      } else {
        // against the current reference at once. No probability exceeds 2^8
        // unless the row sum does, so only then is the tile's maximum taken;
        // where it moved past the threshold the warp computes the tile again
        // (every thread takes part: the P stores are warp-collective)
        sum = exp_pass(-m_ref);
        if (__any_sync(0xffffffffu, !(sum <= 256.0f))) {
          const float m_tile = row_max() * c_log2;
          const bool move = m_tile > m_ref + fa::kRescaleThreshold;
          if (__any_sync(0xffffffffu, move)) {
            if (move) {
              alpha = ex2_approx(m_ref - m_tile);
              m_ref = m_tile;
            }
            tmem_store_wait();   // the first pass's stores land before they are overwritten
            sum = exp_pass(-m_ref);
          }
        }
      }
      l = l * alpha + sum;
      if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
        for (int c = 0; c < C::kDim / 32; ++c) {
          uint32_t o[32];
          tmem_load_32x32(t_o + 32u * c, o);
          tmem_load_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_store_32x32(t_o + 32u * c, o);
        }
      }
      tmem_store_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(t));
    }
    if (ok && warp_wait(o_done(t), 0)) {
      tc_fence_after_sync();
      const float inv_l = 1.0f / l;
      uint16_t* out = static_cast<uint16_t*>(args.o) +
                      ((static_cast<int64_t>(b) * args.seq + q_row) * args.heads + h) * C::kDim;
#pragma unroll
      for (int c = 0; c < C::kDim / 32; ++c) {
        uint32_t o[32];
        tmem_load_32x32(t_o + 32u * c, o);
        tmem_load_wait();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = fa::pack2<C::kBf16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        if (q_row < args.seq) {
          uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == fa::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc<1>(tmem_base, C::kTmemCols);
  }
}

}  // namespace gemm_tn_dev

namespace gemm_tn_impl {

namespace {

template <class C>
cudaError_t launch_cfg(const gemm_tn_dev::FlashArgs& args, unsigned grid, cudaStream_t stream) {
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done_mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_tn_dev::flash_attn_fwd_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    done_mask.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(C::kNumThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent_launch_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_tn_dev::flash_attn_fwd_kernel<C>, args);
}

}  // namespace

int flash_attn_rows_per_cta() { return gemm_tn_dev::fa::kTiles * gemm_tn_dev::fa::kBlockM; }

cudaError_t launch_flash_attn(int head_dim, bool bf16, const gemm_tn_dev::FlashArgs& args, unsigned grid,
                              cudaStream_t stream) {
  using namespace gemm_tn_dev::fa;
  if (head_dim == 64)
    return bf16 ? launch_cfg<Cfg<64, true>>(args, grid, stream) : launch_cfg<Cfg<64, false>>(args, grid, stream);
  if (head_dim == 128)
    return bf16 ? launch_cfg<Cfg<128, true>>(args, grid, stream) : launch_cfg<Cfg<128, false>>(args, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gemm_tn_impl
