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
// The sm_103a mapping (one CTA per 128 queries of one (batch, head)):
//   warp 0      TMA producer: Q once, then K_j and V_j into rings of 128-key
//               tiles (64-element boxes, 128-byte swizzle; the 3-D tensor
//               maps {heads*dim, seq, batch} zero-fill rows past seq).
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               score buffers (M = N = 128, K = dim, both operands from shared
//               memory), then O += P_{j-1} V_{j-1} (M = 128, N = dim, K = 128
//               keys) with P read from tensor memory and V through an MN-major
//               shared-memory descriptor (no transpose). O lives in TMEM for
//               the whole walk.
//   warps 2..   softmax, kSplits groups of four warps. Query row r is TMEM
//               lane r; group g owns score columns [g*128/kSplits, ...) and
//               output columns [g*dim/kSplits, ...) of every row, so each row
//               is shared by kSplits threads (one per group, same lane) that
//               exchange their partial row maxima through shared memory and
//               a named barrier. Per key tile a thread loads its scores,
//               stores P = exp2(s * scale * log2e - max), rounded to the input
//               type, into one of two TMEM P buffers (two values per column),
//               rescales its part of the O row in TMEM when needed, and at the
//               end divides by the row sum and stores its output columns.
// While the softmax warps work on S_j, the tensor cores compute S_{j+1}
// and P_{j-1} V_{j-1}. Keeping P in tensor memory keeps it off the shared
// memory bandwidth, which the operand reads of the two products and the TMA
// writes of K and V already load.
//
// Grid order: work units walk the query tiles of a group of heads whose K
// and V fit in L2 together, so the tiles of one head share K and V through
// L2; with the causal mask the heaviest query tiles (the last ones, which walk
// the most keys) of a group start first.
//
// One difference from the section's loop: the reference maximum of a row is
// only moved when a tile's maximum exceeds it by more than 2^8 (then O and the
// row sum are rescaled); otherwise the probabilities are taken against the
// old maximum (values up to 2^8, exact in fp16 and bf16 range). The result is
// the same softmax -- the final division uses the same reference for the
// numerator and the row sum -- with far fewer O rescales.
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
constexpr int kBlockM = 128;       // queries per CTA (TMEM lanes)
constexpr int kBlockN = 128;       // keys per tile
constexpr int kStatusTimeout = 6;  // == GEMM_TN_ERR_TIMEOUT
// log2 of the largest factor by which probabilities may exceed 1 before the
// row's reference maximum is moved
constexpr float kRescaleThreshold = 8.0f;

template <int kDim_, bool kBf16_, int kSplits_>
struct Cfg {
  static constexpr int kDim = kDim_;
  static constexpr bool kBf16 = kBf16_;
  static constexpr int kSplits = kSplits_;                // softmax warp groups sharing each row
  static constexpr int kCols = kBlockN / kSplits;         // score columns per softmax thread
  static constexpr int kOCols = kDim / kSplits;           // output columns per softmax thread
  static constexpr int kNumThreads = 64 + 128 * kSplits;
  // registers per thread for one CTA per SM: each of the four SM
  // sub-partitions holds 16384 registers and ceil(warps / 4) of the warps
  // (multiples of 8 per thread)
  static constexpr int kMaxRegs = (16384 / 32 / ((kNumThreads / 32 + 3) / 4)) / 8 * 8;
  static constexpr int kDimBoxes = kDim / 64;             // 64-element (128-byte) boxes across dim
  static constexpr uint32_t kBoxBytes = 128u * 128u;      // 128 rows x 128 bytes
  static constexpr uint32_t kTileBytes = kDimBoxes * kBoxBytes;
  static constexpr int kKStages = kDim == 64 ? 4 : 3;     // K ring depth
  static constexpr int kVStages = kDim == 64 ? 4 : 2;     // V ring depth
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
  static constexpr uint32_t kOffRed = kOffV + kVStages * kTileBytes;   // [2][kSplits][128] fp32 partials
  static constexpr uint32_t kOffBar = kOffRed + 2u * kSplits * 128u * 4u;
  // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2], s_empty[2], p_full, o_done, drain
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 4 + 3;
  static constexpr uint32_t kOffTmemSlot = kOffBar + 8u * kNumBars;
  static constexpr uint32_t kOffAbort = kOffTmemSlot + 4u;
  static constexpr uint32_t kSmemBytes = kOffAbort + 4u + 1024u;   // + slack to align the base to 1024
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;      // two 128-column fp32 score buffers
  static constexpr uint32_t kColO = 256;    // dim columns of output accumulator
  static constexpr uint32_t kColP = 384;    // two 64-column buffers of P (two 16-bit values per column)
  static constexpr uint32_t kIdescS = mma_idesc_f16(kBf16, kBlockM, kBlockN, false);
  static constexpr uint32_t kIdescO = mma_idesc_f16(kBf16, kBlockM, kDim, true);
  static_assert(kDim == 64 || kDim == 128, "head dim 64 or 128");
  static_assert(kSplits == 2 || kSplits == 4, "two or four softmax groups");
  static_assert(kCols % 32 == 0 && kOCols % 16 == 0, "TMEM access widths");
  static_assert(kSmemBytes <= 227u * 1024u, "shared memory budget");
  static_assert(kColO + kDim <= kColP && kColP + 128 <= kTmemCols, "TMEM budget");
};

struct Watch {
  const FlashArgs* args;
  volatile uint32_t* abort_flag;

  // Wait for the phase of `bar` with parity `parity`; false on timeout or when
  // another role has given up.
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (mbar_try_wait<false>(bar, parity)) return true;
    const uint64_t deadline = globaltimer_ns() + args->timeout_ns;
    while (true) {
      if (mbar_try_wait<false>(bar, parity)) return true;
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
    while (!mbar_try_wait<false>(bar, parity)) {
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

  // work unit: groups of args.head_group (batch, head) pairs, query tiles
  // of a group interleaved across its heads, heaviest first when causal
  const int n_q = args.num_q_tiles;
  const int bh_count = args.batch * args.heads;
  const int group = static_cast<int>(blockIdx.x) / (args.head_group * n_q);
  const int first_bh = group * args.head_group;
  const int heads_here = min(args.head_group, bh_count - first_bh);
  const int rem = static_cast<int>(blockIdx.x) - group * args.head_group * n_q;
  const int unit_rank = rem / heads_here;
  const int bh = first_bh + rem % heads_here;
  const int qb = args.causal ? n_q - 1 - unit_rank : unit_rank;
  const int b = bh / args.heads;
  const int h = bh % args.heads;
  const int q0 = qb * fa::kBlockM;
  const int key_end = args.causal ? min(args.seq, q0 + fa::kBlockM) : args.seq;
  const int n_kv = (key_end + fa::kBlockN - 1) / fa::kBlockN;
  const int x0 = h * C::kDim;   // column of this head in the {heads*dim, seq, batch} maps

  auto k_tile = [&](int s) { return base + C::kOffK + s * C::kTileBytes; };
  auto v_tile = [&](int s) { return base + C::kOffV + s * C::kTileBytes; };
  auto bar = [&](int i) { return base + C::kOffBar + 8u * i; };
  constexpr int kVBar = 1 + 2 * C::kKStages;                 // first V barrier
  constexpr int kSBar = kVBar + 2 * C::kVStages;              // first score barrier
  const uint32_t q_full = bar(0);
  auto k_full = [&](int s) { return bar(1 + s); };
  auto k_empty = [&](int s) { return bar(1 + C::kKStages + s); };
  auto v_full = [&](int s) { return bar(kVBar + s); };
  auto v_empty = [&](int s) { return bar(kVBar + C::kVStages + s); };
  auto s_full = [&](int i) { return bar(kSBar + i); };
  auto s_empty = [&](int i) { return bar(kSBar + 2 + i); };
  const uint32_t p_full = bar(kSBar + 4);
  const uint32_t o_done = bar(kSBar + 5);
  const uint32_t drain_bar = bar(kSBar + 6);
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(s_empty(i), 4 * C::kSplits);   // one arrival per softmax warp
    }
    mbar_init(p_full, 4 * C::kSplits);
    mbar_init(o_done, 1);
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
  const fa::Watch wd{&args, abort_flag};

  if (warp == fa::kProducerWarp) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int issued_k[C::kKStages], issued_v[C::kVStages];
      for (int s = 0; s < C::kKStages; ++s) issued_k[s] = -1;
      for (int s = 0; s < C::kVStages; ++s) issued_v[s] = -1;
      mbar_arrive_expect_tx(q_full, C::kTileBytes);
      for (int c = 0; c < C::kDimBoxes; ++c)
        tma_load_3d(&args.tmap_q, base + C::kOffQ + c * C::kBoxBytes, q_full, x0 + 64 * c, q0, b);
      const bool drop_here = blockIdx.x == 0;
      for (int j = 0; j < n_kv; ++j) {
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
      bool ok = wd.wait(q_full, 0);
      tc_fence_after_sync();
      const uint32_t q_base = base + C::kOffQ;
      const uint32_t t_o = tmem_base + C::kColO;
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {
          // S_j = Q K_j^T into score buffer j & 1
          const int s = j % C::kKStages;
          const uint32_t ph = static_cast<uint32_t>(j / C::kKStages) & 1u;
          if (!wd.wait(k_full(s), ph) || !wd.wait(s_empty(j & 1), ((static_cast<uint32_t>(j) >> 1) & 1u) ^ 1u)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t t_s = tmem_base + C::kColS + 128u * static_cast<uint32_t>(j & 1);
#pragma unroll
          for (int c = 0; c < C::kDimBoxes; ++c) {
            const uint64_t a_desc = sw128_kmajor_desc(q_base + c * C::kBoxBytes);
            const uint64_t b_desc = sw128_kmajor_desc(k_tile(s) + c * C::kBoxBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)   // 16 elements of dim = 32 bytes = 2 descriptor units
              mma_f16<1>(t_s, a_desc + 2u * kk, b_desc + 2u * kk, C::kIdescS, (c | kk) != 0 ? 1u : 0u);
          }
          mma_commit(k_empty(s));
          mma_commit(s_full(j & 1));
        }
        if (j >= 1) {
          // O += P_{j-1} V_{j-1}: P from its TMEM buffer, V through an MN-major descriptor
          const int i = j - 1;
          const int s = i % C::kVStages;
          const uint32_t ph = static_cast<uint32_t>(i / C::kVStages) & 1u;
          if (!wd.wait(p_full, static_cast<uint32_t>(i) & 1u) || !wd.wait(v_full(s), ph)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t v_desc = sw128_mnmajor_desc(v_tile(s), C::kBoxBytes);
          const uint32_t t_p = tmem_base + C::kColP + 64u * static_cast<uint32_t>(i & 1);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // 16 keys: 8 columns of P; 16 rows of 128 bytes of V
            mma_f16_tmem_a(t_o, t_p + 8u * kk, v_desc + ((static_cast<uint32_t>(kk) * 2048u) >> 4), C::kIdescO,
                           (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(v_empty(s));
          mma_commit(o_done);
        }
      }
      // every MMA issued here must finish before TMEM is freed
      mma_commit(drain_bar);
      wd.drain(drain_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int g = (static_cast<int>(warp) - fa::kFirstSoftmaxWarp) >> 2;   // column group
    const uint32_t quarter = warp & 3u;                                    // TMEM lanes 32*quarter ..
    const int r = static_cast<int>(quarter * 32u + lane);                  // row of the tile
    const int q_row = q0 + r;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const int col0 = g * C::kCols;                                         // first score column
    const uint32_t t_o = tmem_base + lane_off + C::kColO + static_cast<uint32_t>(g * C::kOCols);
    // P of this thread's keys: kCols / 2 columns of a TMEM P buffer
    const uint32_t t_p = tmem_base + lane_off + C::kColP + static_cast<uint32_t>(col0 / 2);
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    auto red_at = [&](int buf, int grp) -> float& { return red[(buf * C::kSplits + grp) * 128 + r]; };
    // the kSplits warps holding the same 32 rows meet at named barrier 1 + quarter
    const uint32_t bar_id = 1u + quarter;
    constexpr uint32_t kBarCount = 32u * C::kSplits;
    const float c_log2 = args.scale_log2;
    // keys this row may see: k < limit
    const int limit = args.causal ? min(q_row + 1, args.seq) : args.seq;
    // waits with a warp-uniform outcome: the tcgen05 loads and stores that
    // follow them are warp-collective
    auto warp_wait = [&](uint32_t bar_addr, uint32_t parity) {
      return __all_sync(0xffffffffu, wd.wait(bar_addr, parity));
    };
    float m_ref = -INFINITY;   // reference maximum, in units of scale * log2e
    float l = 0.0f;            // this thread's part of the row sum, against m_ref
    bool ok = true;
    // Every iteration passes the exchange barrier exactly once, also after a
    // failed wait (the work is then skipped), so no thread can be left
    // waiting at a named barrier for a peer that gave up.
    for (int j = 0; j < n_kv; ++j) {
      const bool live = ok && warp_wait(s_full(j & 1), (static_cast<uint32_t>(j) >> 1) & 1u);
      float sv[C::kCols];
      float mx = -INFINITY;
      if (live) {
        tc_fence_after_sync();
        const uint32_t t_s = tmem_base + lane_off + C::kColS + 128u * static_cast<uint32_t>(j & 1) +
                             static_cast<uint32_t>(col0);
        uint32_t sr[C::kCols / 32][32];
#pragma unroll
        for (int c = 0; c < C::kCols / 32; ++c) tmem_load_32x32(t_s + 32u * c, sr[c]);
        tmem_load_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty(j & 1));
#pragma unroll
        for (int c = 0; c < C::kCols / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[c * 32 + e] = __uint_as_float(sr[c][e]);
        const int key0 = j * fa::kBlockN + col0;
        if (key0 + C::kCols > limit) {
#pragma unroll
          for (int e = 0; e < C::kCols; ++e)
            if (key0 + e >= limit) sv[e] = -INFINITY;
        }
        float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
        for (int e = 4; e < C::kCols; e += 4) {
          mx0 = fmaxf(mx0, sv[e]);
          mx1 = fmaxf(mx1, sv[e + 1]);
          mx2 = fmaxf(mx2, sv[e + 2]);
          mx3 = fmaxf(mx3, sv[e + 3]);
        }
        mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      }
      red_at(j & 1, g) = mx;
      named_barrier_sync(bar_id, kBarCount);
      if (!live) {
        ok = false;
        continue;
      }
      float row_max = red_at(j & 1, 0);
#pragma unroll
      for (int gg = 1; gg < C::kSplits; ++gg) row_max = fmaxf(row_max, red_at(j & 1, gg));
      const float m_tile = row_max * c_log2;
      float alpha = 1.0f;
      if (m_tile > m_ref + fa::kRescaleThreshold) {
        alpha = ex2_approx(m_ref - m_tile);   // 0 on the first tile (m_ref = -inf)
        m_ref = m_tile;
      }
      const float neg_m = -m_ref;
      uint32_t pk[C::kCols / 2];
      float sum0 = 0.0f, sum1 = 0.0f, sum2 = 0.0f, sum3 = 0.0f;
#pragma unroll
      for (int e = 0; e < C::kCols / 2; e += 2) {
        const float p0 = ex2_approx(fmaf(sv[2 * e], c_log2, neg_m));
        const float p1 = ex2_approx(fmaf(sv[2 * e + 1], c_log2, neg_m));
        const float p2 = ex2_approx(fmaf(sv[2 * e + 2], c_log2, neg_m));
        const float p3 = ex2_approx(fmaf(sv[2 * e + 3], c_log2, neg_m));
        sum0 += p0;
        sum1 += p1;
        sum2 += p2;
        sum3 += p3;
        pk[e] = fa::pack2<C::kBf16>(p0, p1);
        pk[e + 1] = fa::pack2<C::kBf16>(p2, p3);
      }
      l = l * alpha + ((sum0 + sum1) + (sum2 + sum3));
      // P_j into TMEM buffer j & 1 (its last reader, P_{j-2} V_{j-2}, finished
      // before this thread's previous tile passed its o_done wait)
      if constexpr (C::kCols == 32) {
        tmem_store_32x16(t_p + 64u * static_cast<uint32_t>(j & 1), pk);
      } else {
        tmem_store_32x32(t_p + 64u * static_cast<uint32_t>(j & 1), pk);
      }

      if (j > 0) {
        // P_{j-1} V_{j-1} has finished: O is stable
        if (!warp_wait(o_done, static_cast<uint32_t>(j - 1) & 1u)) {
          ok = false;
          continue;
        }
        tc_fence_after_sync();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
          if constexpr (C::kOCols % 32 == 0) {
#pragma unroll
            for (int c = 0; c < C::kOCols / 32; ++c) {
              uint32_t o[32];
              tmem_load_32x32(t_o + 32u * c, o);
              tmem_load_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_store_32x32(t_o + 32u * c, o);
            }
          } else {
            uint32_t o[16];
            tmem_load_32x16(t_o, o);
            tmem_load_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_store_32x16(t_o, o);
          }
        }
      }
      tmem_store_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // the row sum: add the kSplits parts (every thread passes this barrier)
    red_at(n_kv & 1, g) = l;
    named_barrier_sync(bar_id, kBarCount);
    float l_row = 0.0f;
#pragma unroll
    for (int gg = 0; gg < C::kSplits; ++gg) l_row += red_at(n_kv & 1, gg);
    if (ok && n_kv > 0 && warp_wait(o_done, static_cast<uint32_t>(n_kv - 1) & 1u)) {
      tc_fence_after_sync();
      const float inv_l = 1.0f / l_row;
      uint16_t* out = static_cast<uint16_t*>(args.o) +
                      ((static_cast<int64_t>(b) * args.seq + q_row) * args.heads + h) * C::kDim + g * C::kOCols;
      auto store16 = [&](const uint32_t* o, int col) {   // 16 fp32 columns -> 32 bytes of output
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          w[e] = fa::pack2<C::kBf16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        if (q_row < args.seq) {
          uint4* dst = reinterpret_cast<uint4*>(out + col);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      };
      if constexpr (C::kOCols % 32 == 0) {
#pragma unroll
        for (int c = 0; c < C::kOCols / 32; ++c) {
          uint32_t o[32];
          tmem_load_32x32(t_o + 32u * c, o);
          tmem_load_wait();
          store16(o, 32 * c);
          store16(o + 16, 32 * c + 16);
        }
      } else {
        uint32_t o[16];
        tmem_load_32x16(t_o, o);
        tmem_load_wait();
        store16(o, 0);
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
  gemm_tn_dev::flash_attn_fwd_kernel<C><<<grid, C::kNumThreads, C::kSmemBytes, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_flash_attn(int head_dim, bool bf16, int splits, const gemm_tn_dev::FlashArgs& args, unsigned grid,
                              cudaStream_t stream) {
  using namespace gemm_tn_dev::fa;
  if (splits == 2) {
    if (head_dim == 64)
      return bf16 ? launch_cfg<Cfg<64, true, 2>>(args, grid, stream) : launch_cfg<Cfg<64, false, 2>>(args, grid, stream);
    if (head_dim == 128)
      return bf16 ? launch_cfg<Cfg<128, true, 2>>(args, grid, stream)
                  : launch_cfg<Cfg<128, false, 2>>(args, grid, stream);
  } else if (splits == 4) {
    if (head_dim == 64)
      return bf16 ? launch_cfg<Cfg<64, true, 4>>(args, grid, stream) : launch_cfg<Cfg<64, false, 4>>(args, grid, stream);
    if (head_dim == 128)
      return bf16 ? launch_cfg<Cfg<128, true, 4>>(args, grid, stream)
                  : launch_cfg<Cfg<128, false, 4>>(args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gemm_tn_impl
