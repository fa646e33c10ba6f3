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
// The sm_103a mapping (one CTA per 128 queries of one (batch, head); 6 warps):
//   warp 0      TMA producer: Q once, then K_j and V_j into two rings of
//               128-key tiles (64-element boxes, 128-byte swizzle; the 3-D
//               tensor maps {heads*dim, seq, batch} zero-fill rows past seq).
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               score buffers (M = N = 128, K = dim), then O += P_{j-1} V_{j-1}
//               (M = 128, N = dim, K = 128 keys; V is read through an MN-major
//               descriptor, no transpose). O lives in TMEM for the whole walk.
//   warps 2-5   softmax: thread r owns query row r (TMEM lane r). It loads
//               the 128 scores of its row, updates the row maximum, writes
//               P = exp2(s * scale * log2e - max) rounded to the input type
//               into shared memory (the A operand of the next MMA, 128-byte
//               swizzle), rescales its O row in TMEM when needed, and at the
//               end divides O by the row sum and stores it.
// While the softmax warps work on S_j, the tensor cores compute S_{j+1}
// and P_{j-1} V_{j-1}.
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

constexpr int kNumThreads = 192;   // 6 warps
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kBlockM = 128;       // queries per CTA (TMEM lanes)
constexpr int kBlockN = 128;       // keys per tile
constexpr int kStatusTimeout = 6;  // == GEMM_TN_ERR_TIMEOUT
// log2 of the largest factor by which probabilities may exceed 1 before the
// row's reference maximum is moved
constexpr float kRescaleThreshold = 8.0f;

template <int kDim_, bool kBf16_>
struct Cfg {
  static constexpr int kDim = kDim_;
  static constexpr bool kBf16 = kBf16_;
  static constexpr int kDimBoxes = kDim / 64;             // 64-element (128-byte) boxes across dim
  static constexpr uint32_t kBoxBytes = 128u * 128u;      // 128 rows x 128 bytes
  static constexpr uint32_t kTileBytes = kDimBoxes * kBoxBytes;
  static constexpr int kStages = kDim == 64 ? 4 : 2;      // K and V ring depth
  static constexpr uint32_t kPBytes = 2 * kBoxBytes;      // 128 rows x 128 keys
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
  static constexpr uint32_t kOffP = kOffV + kStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffP + kPBytes;
  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], s_empty[2], p_full, o_done, drain
  static constexpr int kNumBars = 1 + 4 * kStages + 4 + 3;
  static constexpr uint32_t kOffTmemSlot = kOffBar + 8u * kNumBars;
  static constexpr uint32_t kOffAbort = kOffTmemSlot + 4u;
  static constexpr uint32_t kSmemBytes = kOffAbort + 4u + 1024u;   // + slack to align the base to 1024
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;      // two 128-column score buffers
  static constexpr uint32_t kColO = 256;    // dim columns of output accumulator
  static constexpr uint32_t kIdescS = mma_idesc_f16(kBf16, kBlockM, kBlockN, false);
  static constexpr uint32_t kIdescO = mma_idesc_f16(kBf16, kBlockM, kDim, true);
  static_assert(kDim == 64 || kDim == 128, "head dim 64 or 128");
  static_assert(kSmemBytes <= 227u * 1024u, "shared memory budget");
  static_assert(kColO + kDim <= kTmemCols, "TMEM budget");
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
__global__ void __launch_bounds__(fa::kNumThreads, 1) flash_attn_fwd_kernel(const __grid_constant__ FlashArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t base = smem_addr(smem);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  // work unit: heaviest query tiles first when causal (they walk the most keys)
  const int bh_count = args.batch * args.heads;
  const int unit_rank = static_cast<int>(blockIdx.x) / bh_count;
  const int bh = static_cast<int>(blockIdx.x) % bh_count;
  const int qb = args.causal ? args.num_q_tiles - 1 - unit_rank : unit_rank;
  const int b = bh / args.heads;
  const int h = bh % args.heads;
  const int q0 = qb * fa::kBlockM;
  const int key_end = args.causal ? min(args.seq, q0 + fa::kBlockM) : args.seq;
  const int n_kv = (key_end + fa::kBlockN - 1) / fa::kBlockN;
  const int x0 = h * C::kDim;   // column of this head in the {heads*dim, seq, batch} maps

  auto k_tile = [&](int s) { return base + C::kOffK + s * C::kTileBytes; };
  auto v_tile = [&](int s) { return base + C::kOffV + s * C::kTileBytes; };
  auto bar = [&](int i) { return base + C::kOffBar + 8u * i; };
  const uint32_t q_full = bar(0);
  auto k_full = [&](int s) { return bar(1 + s); };
  auto k_empty = [&](int s) { return bar(1 + C::kStages + s); };
  auto v_full = [&](int s) { return bar(1 + 2 * C::kStages + s); };
  auto v_empty = [&](int s) { return bar(1 + 3 * C::kStages + s); };
  auto s_full = [&](int i) { return bar(1 + 4 * C::kStages + i); };
  auto s_empty = [&](int i) { return bar(3 + 4 * C::kStages + i); };
  const uint32_t p_full = bar(5 + 4 * C::kStages);
  const uint32_t o_done = bar(6 + 4 * C::kStages);
  const uint32_t drain_bar = bar(7 + 4 * C::kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffAbort);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(s_empty(i), 4);   // one arrival per softmax warp
    }
    mbar_init(p_full, 4);
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
      int issued_k[C::kStages], issued_v[C::kStages];
      for (int s = 0; s < C::kStages; ++s) issued_k[s] = issued_v[s] = -1;
      mbar_arrive_expect_tx(q_full, C::kTileBytes);
      for (int c = 0; c < C::kDimBoxes; ++c)
        tma_load_3d(&args.tmap_q, base + C::kOffQ + c * C::kBoxBytes, q_full, x0 + 64 * c, q0, b);
      const bool drop_here = blockIdx.x == 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % C::kStages;
        const uint32_t ph = static_cast<uint32_t>(j / C::kStages) & 1u;
        if (!wd.wait(k_empty(s), ph ^ 1u)) break;
        mbar_arrive_expect_tx(k_full(s), C::kTileBytes);
        if (!(drop_here && j == args.drop_load_block)) {
          for (int c = 0; c < C::kDimBoxes; ++c)
            tma_load_3d(&args.tmap_k, k_tile(s) + c * C::kBoxBytes, k_full(s), x0 + 64 * c, j * fa::kBlockN, b);
        }
        issued_k[s] = static_cast<int>(ph);
        if (!wd.wait(v_empty(s), ph ^ 1u)) break;
        mbar_arrive_expect_tx(v_full(s), C::kTileBytes);
        for (int c = 0; c < C::kDimBoxes; ++c)
          tma_load_3d(&args.tmap_v, v_tile(s) + c * C::kBoxBytes, v_full(s), x0 + 64 * c, j * fa::kBlockN, b);
        issued_v[s] = static_cast<int>(ph);
      }
      // Loads may still be landing if another role gave up: wait (bounded)
      // for every phase issued before the CTA may exit.
      wd.drain(q_full, 0);
      for (int s = 0; s < C::kStages; ++s) {
        if (issued_k[s] >= 0) wd.drain(k_full(s), static_cast<uint32_t>(issued_k[s]));
        if (issued_v[s] >= 0) wd.drain(v_full(s), static_cast<uint32_t>(issued_v[s]));
      }
    }
  } else if (warp == fa::kMmaWarp) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      bool ok = wd.wait(q_full, 0);
      tc_fence_after_sync();
      const uint32_t q_base = base + C::kOffQ;
      const uint32_t p_base = base + C::kOffP;
      const uint32_t t_o = tmem_base + C::kColO;
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {
          // S_j = Q K_j^T into score buffer j & 1
          const int s = j % C::kStages;
          const uint32_t ph = static_cast<uint32_t>(j / C::kStages) & 1u;
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
          // O += P_{j-1} V_{j-1}
          const int i = j - 1;
          const int s = i % C::kStages;
          const uint32_t ph = static_cast<uint32_t>(i / C::kStages) & 1u;
          if (!wd.wait(p_full, static_cast<uint32_t>(i) & 1u) || !wd.wait(v_full(s), ph)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t v_desc = sw128_mnmajor_desc(v_tile(s), C::kBoxBytes);
#pragma unroll
          for (int c = 0; c < 2; ++c) {   // keys 64c .. 64c + 63
            const uint64_t a_desc = sw128_kmajor_desc(p_base + c * C::kBoxBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // 16 keys: 32 bytes along a P row; 16 rows of 128 bytes of V
              const uint32_t v_off = (static_cast<uint32_t>(c) * 8192u + static_cast<uint32_t>(kk) * 2048u) >> 4;
              mma_f16<1>(t_o, a_desc + 2u * kk, v_desc + v_off, C::kIdescO, (i > 0 || c > 0 || kk > 0) ? 1u : 0u);
            }
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
    const uint32_t quarter = warp & 3u;                      // TMEM lanes 32*quarter ..
    const int r = static_cast<int>(quarter * 32u + lane);    // row of the tile
    const int q_row = q0 + r;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const uint32_t t_o = tmem_base + lane_off + C::kColO;
    const uint32_t p_row = base + C::kOffP + static_cast<uint32_t>(r) * 128u;
    const uint32_t swz = static_cast<uint32_t>(r) & 7u;
    const float c_log2 = args.scale_log2;
    // keys this row may see: k < limit
    const int limit = args.causal ? min(q_row + 1, args.seq) : args.seq;
    // waits with a warp-uniform outcome: the tcgen05 loads and stores that
    // follow them are warp-collective
    auto warp_wait = [&](uint32_t bar_addr, uint32_t parity) {
      return __all_sync(0xffffffffu, wd.wait(bar_addr, parity));
    };
    float m_ref = -INFINITY;   // reference maximum, in units of scale * log2e
    float l = 0.0f;            // row sum of probabilities against m_ref
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!warp_wait(s_full(j & 1), (static_cast<uint32_t>(j) >> 1) & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t t_s = tmem_base + lane_off + C::kColS + 128u * static_cast<uint32_t>(j & 1);
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_load_32x32(t_s + 32u * c, sr[c]);
      tmem_load_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty(j & 1));

      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) sv[c * 32 + e] = __uint_as_float(sr[c][e]);
      const int key0 = j * fa::kBlockN;
      const bool masked_tile = key0 + fa::kBlockN > args.seq || (args.causal && key0 + fa::kBlockN - 1 > q0);
      if (masked_tile) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (key0 + e >= limit) sv[e] = -INFINITY;
      }
      float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
      for (int e = 4; e < 128; e += 4) {
        mx0 = fmaxf(mx0, sv[e]);
        mx1 = fmaxf(mx1, sv[e + 1]);
        mx2 = fmaxf(mx2, sv[e + 2]);
        mx3 = fmaxf(mx3, sv[e + 3]);
      }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c_log2;
      float alpha = 1.0f;
      if (m_tile > m_ref + fa::kRescaleThreshold) {
        alpha = ex2_approx(m_ref - m_tile);   // 0 on the first tile (m_ref = -inf)
        m_ref = m_tile;
      }
      const float neg_m = -m_ref;
      uint32_t pk[64];
      float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
      for (int e = 0; e < 64; ++e) {
        const float p0 = ex2_approx(fmaf(sv[2 * e], c_log2, neg_m));
        const float p1 = ex2_approx(fmaf(sv[2 * e + 1], c_log2, neg_m));
        sum0 += p0;
        sum1 += p1;
        pk[e] = fa::pack2<C::kBf16>(p0, p1);
      }
      l = l * alpha + (sum0 + sum1);

      if (j > 0) {
        // P_{j-1} V_{j-1} has finished: the P buffer is free and O is stable
        if (!warp_wait(o_done, static_cast<uint32_t>(j - 1) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
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
          tmem_store_wait();
        }
      }
      // P row r: keys 64c + 8k .. + 7 are 16-byte chunk k of row r in box c,
      // stored at chunk k ^ (r & 7) (the 128-byte swizzle the MMA reads)
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_shared_v4(p_row + c * C::kBoxBytes + ((static_cast<uint32_t>(k) ^ swz) << 4), pk[c * 32 + 4 * k],
                       pk[c * 32 + 4 * k + 1], pk[c * 32 + 4 * k + 2], pk[c * 32 + 4 * k + 3]);
      fence_proxy_async_shared();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && n_kv > 0 && warp_wait(o_done, static_cast<uint32_t>(n_kv - 1) & 1u)) {
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
  gemm_tn_dev::flash_attn_fwd_kernel<C><<<grid, gemm_tn_dev::fa::kNumThreads, C::kSmemBytes, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_flash_attn(int head_dim, bool bf16, const gemm_tn_dev::FlashArgs& args, unsigned grid,
                              cudaStream_t stream) {
  using namespace gemm_tn_dev::fa;
  if (head_dim == 64) {
    return bf16 ? launch_cfg<Cfg<64, true>>(args, grid, stream) : launch_cfg<Cfg<64, false>>(args, grid, stream);
  }
  if (head_dim == 128) {
    return bf16 ? launch_cfg<Cfg<128, true>>(args, grid, stream) : launch_cfg<Cfg<128, false>>(args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gemm_tn_impl
