// gemm_tn_api.cu -- the C ABI declared in include/gemm_tn.h: argument
// validation, alignment classification, the frozen configuration table,
// tensor-map encoding and the launch of the sm_103a kernels.
//
// Host flow of one call ("0. A Minimal Hopper Matmul", sections "Kernel Setup"
// and "Running the Kernel": the caller owns A, B, C; the grid covers
// ceil(M / block_m) x ceil(N / block_n) tiles; "TMA: Tensor Memory Access":
// the tensor-map descriptor is built on the host):
//   validate -> (K == 0: zero C) -> classify operand alignment -> repack a
//   misaligned operand into a workspace -> pick a configuration -> encode the
//   tensor maps -> launch the persistent kernel on `stream`.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "flash_attn.h"
#include "gemm_tn.h"
#include "gemm_tn_internal.h"
#include "sm103_gemm_kernel.cuh"

namespace gemm_tn_impl {

cudaError_t launch_gemm_1cta(int id, bool bf16, bool k_pairs, const gemm_tn_dev::GemmArgs& args, int grid,
                             cudaStream_t stream);
int max_resident_1cta(int id, bool bf16);
int smem_bytes_1cta(int id);
cudaError_t launch_gemm_2cta(int id, bool bf16, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream);
int max_resident_2cta(int id, bool bf16);
int smem_bytes_2cta(int id);
cudaError_t launch_gemm_nn(int id, bool bf16, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_gemm_fused(int id, bool bf16, const gemm_tn_dev::GemmArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_gemm_splitk(int splits, bool bf16, bool k_pairs, const gemm_tn_dev::GemmArgs& args, int grid,
                               cudaStream_t stream);
cudaError_t launch_gemm_decode(int splits, int rows, bool bf16, bool k_pairs, const gemm_tn_dev::GemmArgs& args,
                               int grid, cudaStream_t stream);
int decode_rows(int64_t m);
int max_resident_splitk(int splits, bool bf16, int num_sms);
constexpr int kGb300SplitKResidentDefault[3] = {76, 36, 15};
cudaError_t launch_fused_k0(bool bf16, void* c, int64_t ldc, int out_kind, int64_t m, int64_t n, float beta,
                            const float* bias, int activation, int num_sms, cudaStream_t stream);

namespace {

constexpr int kAbiVersion = 100;
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
constexpr int kBlockK = 64;

const ConfigInfo kConfigs[kNumConfigs] = {
    {"1cta_n256", 1, 128, 256, 256, 4, 1, 128},
    {"1cta_n128", 1, 128, 128, 128, 6, 1, 128},
    {"2cta_n256", 2, 256, 256, 128, 6, 1, 128},
    {"2cta_n128", 2, 256, 128, 64, 8, 1, 128},
    {"2cta_n256_mc", 2, 256, 256, 128, 6, 2, 64},
    {"1cta_n128_splitk", 1, 128, 128, 128, 6, 1, 128},
    {"1cta_decode_splitk", 1, 128, 128, 128, 11, 1, 16},
    {"1cta_n64", 1, 128, 64, 64, 8, 1, 128},
};

thread_local int t_last_cuda_error = 0;
std::atomic<uint64_t> g_launch_count{0};

// Count one kernel launch that the runtime accepted.
cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e;
}
thread_local char t_last_message[256] = "";

int fail(int status, const char* what) {
  std::snprintf(t_last_message, sizeof(t_last_message), "%s", what);
  return status;
}

int fail_cuda(cudaError_t e, const char* what) {
  t_last_cuda_error = static_cast<int>(e);
  std::snprintf(t_last_message, sizeof(t_last_message), "%s: %s", what, cudaGetErrorString(e));
  return GEMM_TN_ERR_CUDA;
}

// Configuration the calling thread's last GEMM call launched (-1: none).
thread_local int t_last_config = -1;

// ---------------------------------------------------------------- device facts

struct DeviceFacts {
  bool valid = false;
  int cc_major = 0, cc_minor = 0, num_sms = 0;
  int max_clusters[kNumConfigs][2] = {};   // [config][bf16], 0 = not queried yet
  int splitk_clusters[3][2] = {};           // split-K clusters of 2, 4, 8 CTAs [size][bf16]
};

std::mutex g_device_mutex;
DeviceFacts g_devices[64];

int current_device(DeviceFacts** facts) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return fail(GEMM_TN_ERR_UNSUPPORTED_DEVICE, "no current CUDA device");
  }
  std::lock_guard<std::mutex> lock(g_device_mutex);
  DeviceFacts& f = g_devices[dev];
  if (!f.valid) {
    if (cudaDeviceGetAttribute(&f.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&f.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&f.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return fail(GEMM_TN_ERR_UNSUPPORTED_DEVICE, "cannot query the current device");
    }
    f.valid = true;
  }
  if (f.cc_major != 10 || f.cc_minor != 3) {
    return fail(GEMM_TN_ERR_UNSUPPORTED_DEVICE, "device is not compute capability 10.3 (sm_103a)");
  }
  *facts = &f;
  return GEMM_TN_OK;
}

int resident_clusters(DeviceFacts* f, int cfg, bool bf16) {
  {
    std::lock_guard<std::mutex> lock(g_device_mutex);
    if (f->max_clusters[cfg][bf16] > 0) return f->max_clusters[cfg][bf16];
  }
  // split-K clusters run one tile each (not persistent): one CTA per SM
  const int n = cfg == kCfg1CtaSplitK || cfg == kCfgDecodeSplitK ? f->num_sms
                : kConfigs[cfg].cta_group == 2 ? max_resident_2cta(cfg, bf16)
                                               : max_resident_1cta(cfg, bf16);
  std::lock_guard<std::mutex> lock(g_device_mutex);
  f->max_clusters[cfg][bf16] = n;
  return n;
}

// Resident split-K clusters of 2, 4 and 8 CTAs on the current device (GB300's
// when a query fails).
void splitk_resident(DeviceFacts* f, bool bf16, int out[3]) {
  for (int i = 0; i < 3; ++i) {
    {
      std::lock_guard<std::mutex> lock(g_device_mutex);
      out[i] = f->splitk_clusters[i][bf16];
    }
    if (out[i] > 0) continue;
    int n = max_resident_splitk(2 << i, bf16, f->num_sms);
    if (n <= 0) n = kGb300SplitKResidentDefault[i];
    std::lock_guard<std::mutex> lock(g_device_mutex);
    f->splitk_clusters[i][bf16] = n;
    out[i] = n;
  }
}

// ---------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    } else {
      cudaGetLastError();
    }
  });
  return g_encode;
}

// Row-major [rows, cols] 16-bit matrix with pitch `ld` elements, moved in
// boxes of box_cols x box_rows with the given swizzle. Operands use 64-column
// (128-byte) boxes with the 128-byte swizzle the MMA descriptors expect; C
// uses 32 x 32 boxes with the 64-byte swizzle of the epilogue staging.
// Out-of-range elements read as zero and are not written.
int encode_matrix_map(CUtensorMap* map, bool bf16, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                      int box_cols, int box_rows, CUtensorMapSwizzle swizzle) {
  auto encode = encode_fn();
  if (encode == nullptr) return fail(GEMM_TN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                            const_cast<void*>(ptr), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return fail(GEMM_TN_ERR_CUDA, buf);
  }
  return GEMM_TN_OK;
}

// A K-major [rows, cols] 16-bit matrix (cols a multiple of 64) as a 3-D map
// {64, rows, cols / 64}, moved in boxes of {64, box_rows, 2}: one copy brings
// two 64-column k-blocks, each a 128-byte-swizzled [box_rows x 64] tile, one
// after the other. A box's second k-block past the last reads as zeros.
int encode_kpair_map(CUtensorMap* map, bool bf16, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                     int box_rows) {
  auto encode = encode_fn();
  if (encode == nullptr) return fail(GEMM_TN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 2};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                            const_cast<void*>(ptr), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return fail(GEMM_TN_ERR_CUDA, buf);
  }
  return GEMM_TN_OK;
}

// [batch, seq, heads, dim] 16-bit array as a 3-D map {heads * dim, seq,
// batch}, moved in boxes of {64, 128, 1} (128-byte rows, 128-byte swizzle);
// rows past seq read as zero.
int encode_bshd_map(CUtensorMap* map, bool bf16, const void* ptr, int64_t batch, int64_t seq, int64_t heads,
                    int64_t dim) {
  auto encode = encode_fn();
  if (encode == nullptr) return fail(GEMM_TN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(heads * dim), static_cast<cuuint64_t>(seq),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(heads * dim * 2), static_cast<cuuint64_t>(seq * heads * dim * 2)};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                            const_cast<void*>(ptr), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return fail(GEMM_TN_ERR_CUDA, buf);
  }
  return GEMM_TN_OK;
}

// ---------------------------------------------------------------- validation

bool ranges_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// Bytes spanned by a [rows, cols] matrix with pitch ld (16-bit elements).
uintptr_t span_bytes(int64_t rows, int64_t cols, int64_t ld, int64_t elem_bytes = 2) {
  return static_cast<uintptr_t>(((rows - 1) * ld + cols) * elem_bytes);
}

// Bytes per element of C: the input dtype's 2, or the fused epilogue's
// fp32 / e4m3 output.
int64_t c_elem_bytes(const gemm_tn_epilogue* fused) {
  if (fused == nullptr) return 2;
  return fused->out_dtype == GEMM_TN_OUT_F32 ? 4 : (fused->out_dtype == GEMM_TN_OUT_E4M3 ? 1 : 2);
}

// b_mn: B is [K, N] (N contiguous, ldb >= n) instead of [N, K].
int validate(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda, const void* b, int64_t ldb,
             const void* c, int64_t ldc, bool b_mn = false, int64_t c_elem = 2) {
  if (dtype != GEMM_TN_F16 && dtype != GEMM_TN_BF16) return fail(GEMM_TN_ERR_UNSUPPORTED_DTYPE, "dtype");
  if (m < 0 || n < 0 || k < 0 || m > kMaxDim || n > kMaxDim || k > kMaxDim)
    return fail(GEMM_TN_ERR_INVALID_VALUE, "sizes must be in [0, 2^31)");
  if (m == 0 || n == 0) return GEMM_TN_OK;
  if (c == nullptr) return fail(GEMM_TN_ERR_INVALID_VALUE, "C is NULL");
  if (ldc < n || ldc > kMaxDim * 2) return fail(GEMM_TN_ERR_INVALID_VALUE, "ldc < n");
  if (reinterpret_cast<uintptr_t>(c) % c_elem) return fail(GEMM_TN_ERR_MISALIGNED, "C is not aligned to its element");
  if (k == 0) return GEMM_TN_OK;
  if (a == nullptr || b == nullptr) return fail(GEMM_TN_ERR_INVALID_VALUE, "A or B is NULL");
  if (lda < k || ldb < (b_mn ? n : k) || lda > kMaxDim * 2 || ldb > kMaxDim * 2)
    return fail(GEMM_TN_ERR_INVALID_VALUE, b_mn ? "lda < k or ldb < n" : "lda or ldb < k");
  if (reinterpret_cast<uintptr_t>(a) % 2 || reinterpret_cast<uintptr_t>(b) % 2)
    return fail(GEMM_TN_ERR_MISALIGNED, "A or B is not 2-byte aligned");
  const uintptr_t c0 = reinterpret_cast<uintptr_t>(c), c1 = c0 + span_bytes(m, n, ldc, c_elem);
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), a1 = a0 + span_bytes(m, k, lda);
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(b), b1 = b0 + (b_mn ? span_bytes(k, n, ldb) : span_bytes(n, k, ldb));
  if (ranges_overlap(c0, c1, a0, a1) || ranges_overlap(c0, c1, b0, b1))
    return fail(GEMM_TN_ERR_INVALID_VALUE, "C overlaps A or B");
  return GEMM_TN_OK;
}

// TMA wants a 16-byte-aligned base and a row pitch that is a multiple of 16 bytes.
bool tma_compatible(const void* p, int64_t ld) {
  return reinterpret_cast<uintptr_t>(p) % 16 == 0 && ld % 8 == 0;
}

// Whether `p` is device memory that lives on device `dev` (not host memory,
// managed memory or another GPU's memory reached through peer access).
bool memory_of_device(const void* p, int dev) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

// The multicast configuration (2cta_n256_mc) has one CTA load a half-tile of A
// for two CTA pairs with a cluster-multicast TMA load. It may read only this
// GPU's own memory: both operands must be device memory of the current device.
// Any other pointer (peer, host-mapped, managed) runs the plain pair kernel.
bool multicast_source_ok(const void* a, const void* b) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return memory_of_device(a, dev) && memory_of_device(b, dev);
}

int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }

// ---------------------------------------------------------------- configuration

int parse_forced_config() {
  const char* s = std::getenv("GEMM_TN_FORCE_CONFIG");
  if (s == nullptr || *s == '\0') return -1;
  for (int i = 0; i < kNumConfigs; ++i)
    if (std::strcmp(s, kConfigs[i].name) == 0) return i;
  char* end = nullptr;
  const long v = std::strtol(s, &end, 10);
  if (end != s && *end == '\0' && v >= 0 && v < kNumConfigs) return static_cast<int>(v);
  return -1;
}

// The frozen table, from measurements on GB300.
//  * M <= 128: single-CTA 128 x 128 tiles, so the N dimension alone supplies
//    the tiles (bf16 128 x 16384 x 16384: 5.3 TB/s vs 4.9 for pair tiles).
//  * Otherwise 256 x 256 tiles on CTA pairs (bf16 8192^3: 1698 TFLOP/s vs 1565
//    for single-CTA 128 x 256 tiles), either as plain pairs (76 resident on
//    GB300) or as 4-CTA clusters of two pairs sharing A through multicast (36
//    resident: 144 of the 152 SMs). A multicast cluster streams ~5% more work
//    per SM (fp16 4096^3: 1534 vs 1503 TFLOP/s; fp16 3001 x 5003 x 4097: 857 vs
//    741), so it is chosen when its rounds of tiles, discounted by that 5%,
//    are fewer than the pairs' rounds (bf16 8192^3: 15 rounds vs 14, so pairs).
// K splits of the split-K configuration for an M x N x K problem (0: not
// worth it). With fewer 128 x 128 tiles than half the SMs, each tile's K is
// cut over a cluster of S CTAs, S the largest of 8, 4, 2 whose clusters are
// all resident at once (resident[0..2]: clusters of 2, 4, 8 CTAs; GB300: 76,
// 36, 15) and that leaves enough k-blocks per CTA: 4 for S = 2 and 8, 2 for
// S = 4 (4 for the decode kernel's M <= 32). Measured on GB300 (CUDA graphs, us per call, no split -> split):
// 128 x 1024 x 4096 19.8 -> 6.9 (S = 8), 64 x 2048 x 8192 38.5 -> 12.2 (S = 4;
// 16 clusters of 8 do not fit at once and took 17.2), 1024 x 1024 x 8192 39.5
// -> 20.9 (S = 2); 256^3 (4 k-blocks) stays whole. With 8 to 15 k-blocks S = 4
// beat S = 2 on every shape tried (S = 2 -> 4: 256 x 256 x 512 5.64 -> 4.85,
// 512 x 512 x 896 6.67 -> 5.43, 768^3 6.36 -> 5.95, 640 x 640 x 512 5.74 ->
// 5.33), and S = 2 was at times slower than no split (5.34 and 5.43 there).
// GEMM_TN_SPLITK=<S> forces S (0 turns it off).
int splitk_factor(int64_t m, int64_t n, int64_t k, int sms, const int resident[3]) {
  const int64_t tiles = ((m + 127) / 128) * ((n + 127) / 128);
  const int64_t kb = (k + 63) / 64;
  const char* s = std::getenv("GEMM_TN_SPLITK");
  if (s != nullptr && *s != '\0') {
    const long v = std::strtol(s, nullptr, 10);
    if (v == 0) return 0;
    if ((v == 2 || v == 4 || v == 8) && v <= kb) return static_cast<int>(v);
  }
  if (tiles * 2 > sms) return 0;
  const int splits_of[3] = {2, 4, 8};
  // the 2-k-block 4-way split was measured with the 128 x 128 split-K kernel
  // only; the decode kernel (M <= 32) keeps 4 k-blocks per CTA
  const int min_kb_per_cta[3] = {4, m <= 32 ? 4 : 2, 4};
  for (int i = 2; i >= 0; --i)
    if (tiles <= resident[i] && kb >= min_kb_per_cta[i] * splits_of[i]) return splits_of[i];
  return 0;
}

// The K split a split-K configuration runs with: splitk_factor's choice, or
// for a forced split-K configuration the largest split that K allows; 0 when
// K cannot be cut (the call then runs whole 128 x 128 tiles) or B is [K, N].
int resolve_splits(int64_t m, int64_t n, int64_t k, bool b_mn, int sms, const int resident[3]) {
  if (b_mn) return 0;
  int splits = splitk_factor(m, n, k, sms, resident);
  for (int s : {8, 4, 2})
    if (splits == 0 && s <= (k + kBlockK - 1) / kBlockK) splits = s;
  return splits >= 2 ? splits : 0;
}

int choose_config(int64_t m, int64_t n, int64_t k, int resident_pairs = 76, int resident_quads = 36,
                  const int* splitk_resident = kGb300SplitKResidentDefault) {
  const int forced = parse_forced_config();
  if (forced >= 0) return forced;
  // few output tiles: split K over a cluster (with at most 32 rows of A, B's
  // rows take the MMA's M side) -- unless K is short and 128 x 64 tiles,
  // which move two k-blocks per copy when K is a multiple of 64, fit in one
  // round of the SMs: then the split's partial-sum exchange costs more than
  // it saves (GB300, us per call in CUDA graphs, 1cta_n64 vs the K split:
  // 256 x 256 x 512 4.21 vs 4.62 at S = 4, 512^3 4.41 vs 4.93 at S = 4, 1024^3
  // 5.92 vs 6.37 at S = 2). Longer K, or a wider split, keeps the split.
  const int splits = splitk_factor(m, n, k, 2 * resident_pairs, splitk_resident);
  if (splits > 1) {
    const int64_t kb = (k + 63) / 64;
    const int64_t n64_tiles = ((m + 127) / 128) * ((n + 63) / 64);
    const bool short_k = m > 128 && k % 64 == 0 && n64_tiles <= 2 * static_cast<int64_t>(resident_pairs) &&
                         (kb <= 8 || (kb <= 16 && splits == 2));
    if (!short_k) return m <= 32 ? kCfgDecodeSplitK : kCfg1CtaSplitK;
    return kCfg1CtaN64;
  }
  // Tiny problems: 128 x 64 tiles while they fill at most half the SMs, so
  // more SMs share the operand loads and each epilogue is half as long
  // (GB300, us per call in CUDA graphs, 1cta_n64 vs 1cta_n128: 256^3 3.90
  // vs 4.29, 384 x 384 x 256 4.01 vs 4.21; with 256 tiles of 128 x 64 at
  // 1024 x 2048 x 1024 it took 14.2 against 7.9).
  if (((m + 127) / 128) * ((n + 63) / 64) <= static_cast<int64_t>(resident_pairs)) return kCfg1CtaN64;
  if (m <= 128) return kCfg1CtaN128;
  // One round of single-CTA 128 x 128 tiles: every SM gets at most one tile,
  // and a 128 x 128 tile is half the work of a pair's 256 x 256 (GB300, us
  // per call in CUDA graphs, 1cta_n128 vs the pair / cluster choice: 256^3
  // 4.31 vs 4.52, 1536 x 1536 x 256 4.52 vs 6.58, 1536 x 1536 x 2048 12.4 vs
  // 14.5, 1024 x 2048 x 4096 20.9 vs 23.0).
  if (((m + 127) / 128) * ((n + 127) / 128) <= 2 * static_cast<int64_t>(resident_pairs)) return kCfg1CtaN128;
  // One round of single-CTA 128 x 256 tiles, K up to 4096: the same work per
  // SM as pair tiles without the pairs' cross-CTA hand-offs (2048^2 x 512 6.8
  // vs 8.5 us, 2048^3 14.1 vs 15.5, 2304 x 2048 x 4096 22.9 vs 24.7). Longer K
  // favours the pairs, whose CTAs stream 32 KiB per k-block against 48 KiB
  // (2048^2 x 8192: 50.4 vs 41.9).
  if (((m + 127) / 128) * ((n + 255) / 256) <= 2 * static_cast<int64_t>(resident_pairs) && k <= 4096)
    return kCfg1CtaN256;
  const int64_t tile_rows = (m + 255) / 256;
  const int64_t pair_tiles = tile_rows * ((n + 255) / 256);
  const int64_t quad_tiles = tile_rows * ((n + 511) / 512);
  const double pair_rounds = static_cast<double>((pair_tiles + resident_pairs - 1) / std::max(resident_pairs, 1));
  const double quad_rounds =
      static_cast<double>((quad_tiles + resident_quads - 1) / std::max(resident_quads, 1)) / 1.05;
  return quad_rounds < pair_rounds ? kCfg2CtaN256Mc : kCfg2CtaN256;
}

// GEMM_TN_EPILOGUE=direct forces the predicated element-store epilogue even
// when C could be written through the TMA (used to test both paths).
bool force_direct_epilogue() {
  const char* s = std::getenv("GEMM_TN_EPILOGUE");
  return s != nullptr && std::strcmp(s, "direct") == 0;
}

// Test hook: GEMM_TN_TEST_DROP_LOAD=<k-block> makes each CTA's producer skip
// the loads of that k-block of its first tile, so the MMA issuer's bounded
// wait on it expires and the watchdog path runs (no fault is involved).
int test_drop_load_kb() {
  const char* s = std::getenv("GEMM_TN_TEST_DROP_LOAD");
  if (s == nullptr || *s == '\0') return -1;
  char* end = nullptr;
  const long v = std::strtol(s, &end, 10);
  return (end != s && v >= 0 && v < INT32_MAX) ? static_cast<int>(v) : -1;
}

uint64_t watchdog_ns() {
  const char* s = std::getenv("GEMM_TN_WATCHDOG_MS");
  long ms = 4000;
  if (s != nullptr && *s != '\0') {
    char* end = nullptr;
    const long v = std::strtol(s, &end, 10);
    if (end != s && v > 0) ms = v;
  }
  return static_cast<uint64_t>(ms) * 1000000ull;
}

// ---------------------------------------------------------------- workspace pool
//
// Stream-ordered workspaces (padded copies of misaligned operands, stream-K
// partials and flags) come from a memory pool the library creates once per
// device and that keeps its memory between calls: with the device's default
// pool, whose memory goes back to the system at every synchronisation, a call
// after a synchronisation waited for fresh memory to be mapped (bf16 8192^3
// with a synchronisation after each call: 672 against 580 us on the device).
// gemm_tn_trim_workspace returns the unused part.
std::mutex g_ws_pool_mutex;
cudaMemPool_t g_ws_pool[64] = {};

// The workspace pool of device `dev`, created on first use (a failed
// creation is retried by the next call).
cudaError_t workspace_pool(int dev, cudaMemPool_t* out) {
  std::lock_guard<std::mutex> lock(g_ws_pool_mutex);
  if (g_ws_pool[dev] == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    cudaError_t e = cudaMemPoolCreate(&pool, &props);
    if (e == cudaSuccess) {
      uint64_t keep = UINT64_MAX;
      e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
      if (e != cudaSuccess) cudaMemPoolDestroy(pool);
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e;
    }
    g_ws_pool[dev] = pool;
  }
  *out = g_ws_pool[dev];
  return cudaSuccess;
}

// fixed_scratch: nullptr = workspace from the library's pool (the normal
// path); otherwise a caller-designated device buffer of fixed_scratch_bytes
// that is used instead and never freed (gemm_tn_ex_noalloc).
// How the tiles of one call are shared out over the grid's workers (CTA
// pairs or single CTAs). Whole waves of tiles go data-parallel; when the last
// wave would leave workers idle, the final `clusters + remainder` tiles are
// split by k-block iterations into one contiguous range per worker, each at
// least one tile long, so every worker finishes at about the same time
// ("Tiling a matmul", "Where it breaks": stream-K keeps all SMs busy). With
// fewer tiles than workers, the whole problem is split that way, at least
// kMinSkIters k-blocks per worker.
struct WorkPlan {
  int workers;
  int64_t dp_tiles;
  int64_t sk_iters;
  int sk_workers;   // workers 0 .. sk_workers - 1 share the stream-K iterations
};

constexpr int64_t kMinSkIters = 8;

WorkPlan plan_work(int64_t tiles, int64_t k_blocks, int clusters, int stream_k) {
  WorkPlan p{static_cast<int>(std::min<int64_t>(tiles, clusters)), tiles, 0, 0};
  if (stream_k == 0) return p;
  if (stream_k < 0) {
    // the default: problems of at least one full wave whose last wave is
    // partial cut that wave's tiles into equal k-ranges (mode 3), or, when
    // they are too many for two parts each, spread them over all workers
    // (mode 2). Measured on GB300 against whole tiles with the N cut of the
    // last wave (tail split), us per call: bf16 8192^3 566 -> 552 (mode 3),
    // fp16 4096^3 86.8 -> 84.6 (mode 2), fp16 3001 x 5003 x 4097 119.9 ->
    // 113.7 (mode 3). Fewer tiles than workers keep whole tiles.
    if (tiles < clusters || tiles % clusters == 0) return p;
    const int64_t rem = tiles % clusters;
    stream_k = std::min<int64_t>(clusters / rem, k_blocks / kMinSkIters) >= 2 ? 3 : 2;
  }
  if (tiles >= clusters) {
    const int64_t rem = tiles % clusters;
    if (rem == 0) return p;
    // mode 3: each tile of the partial wave is cut into s equal k-ranges, s =
    // the most parts that give every worker at most one (and each part at
    // least kMinSkIters k-blocks); worker t * s + q takes part q of cut tile
    // t, so the parts running together read the same k-range of tiles that
    // share rows of A or B, and one wave's worth of work is spread over all
    // but clusters - rem * s workers
    if (stream_k == 3) {
      const int64_t s = std::min<int64_t>(clusters / rem, k_blocks / kMinSkIters);
      if (s < 2) return p;
      p.workers = clusters;
      p.dp_tiles = tiles - rem;
      p.sk_iters = rem * k_blocks;
      p.sk_workers = static_cast<int>(rem * s);
      return p;
    }
    // mode 2: only the partial wave's tiles are split (each across about
    // clusters / rem workers), when that leaves at least kMinSkIters k-blocks
    // per worker
    if (stream_k == 2 && rem * k_blocks >= clusters * kMinSkIters) {
      p.workers = clusters;
      p.dp_tiles = tiles - rem;
      p.sk_iters = rem * k_blocks;
      p.sk_workers = clusters;
      return p;
    }
    if (stream_k != 1) return p;
    const int64_t sk_tiles = rem + clusters;
    p.workers = clusters;
    p.dp_tiles = tiles - sk_tiles;
    p.sk_iters = sk_tiles * k_blocks;
    p.sk_workers = clusters;
    return p;
  }
  const int64_t iters = tiles * k_blocks;
  const int64_t w = std::min<int64_t>(clusters, iters / kMinSkIters);
  if (w > tiles) {
    p.workers = static_cast<int>(w);
    p.dp_tiles = 0;
    p.sk_iters = iters;
    p.sk_workers = p.workers;
  }
  return p;
}

// The stream-K tail is the default for a partial last wave (plan_work). Its
// fp32 partial rows go out and come back as 512-byte warp-wide accesses, and
// the contributors' flags carry a per-launch value, so no clearing pass runs
// before the GEMM; with 16-byte-per-row accesses and a memset of the flags
// it had measured slower than whole tiles (fp16 4096^3: 105 against 88.6 us).
// Tail split (used when the stream-K tail is not, e.g. in the no-alloc entry
// point or with GEMM_TN_STREAMK=0): when the tiles leave a last, partial wave, cut each of its
// tiles into `split` sub-tiles along N (2 or 4, keeping N >= 64 per MMA) so
// that wave has up to `split` times as many, shorter units for the same
// workers. Returns the split factor (1: none) and the first cut tile.
// GEMM_TN_TAIL_SPLIT=0 turns it off; =force cuts the last wave whatever the
// number of full waves before it (measurements).

int tail_split(const ConfigInfo& cfg, int64_t tiles, int clusters, int64_t* split_begin, bool b_mn) {
  *split_begin = tiles;
  const char* env = std::getenv("GEMM_TN_TAIL_SPLIT");
  if (env != nullptr && std::strcmp(env, "0") == 0) return 1;
  const bool forced = env != nullptr && std::strcmp(env, "force") == 0;   // any number of full waves
  const int64_t full = tiles >= clusters ? tiles - tiles % clusters : 0;
  const int64_t last = tiles - full;
  if (last == 0) return 1;
  // The split-capable kernel runs every round ~1% slower, so a cut last wave
  // pays only when it is a large share of the work: at most 4 full waves
  // before it (bf16 8192^3, 13 full waves: -1.3 to -1.8% with the cut; fp16
  // 3001 x 5003 x 4097, 3: +4.4%). Running the cut tiles as a second launch
  // after the full waves, with the plain kernel for those, measured worse
  // still (fp16 3001 x 5003 x 4097: 120 against 112 us; bf16 8192^3: +2-3%):
  // the second launch waits for the whole first grid and starts cold.
  if (full / clusters > 4 && !forced) return 1;
  for (int s : {4, 2}) {
    if (cfg.block_n / s >= 64 && (cfg.b_rows / s) % (b_mn ? 64 : 8) == 0 && last * s <= clusters) {
      *split_begin = full;
      return s;
    }
  }
  return 1;
}

// GEMM_TN_STREAMK selects the stream-K mode: unset, the default choice of
// plan_work (-1); 0 whole tiles only; 1 the last partial wave and one full
// wave spread over all workers; 2 only the partial wave's tiles, over all
// workers; 3 each partial-wave tile cut into equal k-ranges, one per worker.
int stream_k_mode() {
  const char* s = std::getenv("GEMM_TN_STREAMK");
  if (s == nullptr || *s == '\0') return -1;
  if (std::strcmp(s, "1") == 0) return 1;
  if (std::strcmp(s, "2") == 0) return 2;
  if (std::strcmp(s, "3") == 0) return 3;
  return 0;
}

// Flag value of one stream-K launch: a tag in the high word and a per-process
// launch counter in the low word. Each launch's flags start as whatever the
// workspace held (no clearing pass): earlier launches wrote smaller counters,
// and a contributor stores this launch's value only once its partial rows are
// written.
std::atomic<uint64_t> g_flag_counter{0};
uint64_t next_flag_epoch() {
  return (0x5EED5EEDull << 32) | ((g_flag_counter.fetch_add(1, std::memory_order_relaxed) + 1) & 0xFFFFFFFFull);
}

// K rotation and evict-first B loads for problems with one row of tiles.
// There every tile streams its own rows of B once (an intensity of at most
// ~M FLOP/B, under the ridge), and with all tiles at the same K offset the
// concurrent reads, a row pitch apart, crowd few DRAM banks: bf16 128 x 16384
// x 16384 measured 5.43 TB/s in the plain order and 5.94 TB/s rotated. With
// several rows of tiles the grouped raster wants tiles to read shared rows of
// A and B at the same time, so the order stays plain. GEMM_TN_K_ROTATE=0/1
// overrides the choice (tests and experiments).
bool k_rotation_on(int64_t num_m_tiles) {
  const char* s = std::getenv("GEMM_TN_K_ROTATE");
  if (s != nullptr && *s != '\0') return std::strcmp(s, "0") != 0;
  return num_m_tiles == 1;
}

// Multiply-and-shift constants for dividing by d (1 <= d < 2^31); see FastDiv.
gemm_tn_dev::FastDiv make_fast_div(int64_t d) {
  uint32_t l = 0;
  while ((int64_t{1} << l) < d) ++l;
  const uint64_t mul = ((uint64_t{1} << 32) * ((uint64_t{1} << l) - static_cast<uint64_t>(d))) /
                           static_cast<uint64_t>(d) + 1;
  return gemm_tn_dev::FastDiv{static_cast<uint32_t>(mul), l};
}

// Tile rows per rasterization group: tiles in flight together then share
// about 2048 rows of A and the matching columns of B in L2.
// GEMM_TN_GROUP_M overrides it (tuning experiments).
int group_rows(const ConfigInfo& cfg) {
  const char* s = std::getenv("GEMM_TN_GROUP_M");
  if (s != nullptr && *s != '\0') {
    const long v = std::strtol(s, nullptr, 10);
    if (v > 0 && v < 65536) return static_cast<int>(v);
  }
  return cfg.cta_group == 2 ? 8 : 16;
}

int run_gemm(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda, const void* b, int64_t ldb,
             void* c, int64_t ldc, int* d_status, cudaStream_t stream, int drop_load_kb,
             void* fixed_scratch = nullptr, size_t fixed_scratch_bytes = 0, bool b_mn = false,
             const gemm_tn_epilogue* fused = nullptr) {
  t_last_cuda_error = 0;
  t_last_message[0] = '\0';
  t_last_config = -1;
  int st = validate(dtype, m, n, k, a, lda, b, ldb, c, ldc, b_mn, c_elem_bytes(fused));
  if (st != GEMM_TN_OK) return st;
  if (m == 0 || n == 0) return GEMM_TN_OK;
  DeviceFacts* dev = nullptr;
  st = current_device(&dev);
  if (st != GEMM_TN_OK) return st;

  // C's element type in the fused epilogue: 0 the input dtype, 1 fp32, 2 e4m3
  const int out_kind = fused == nullptr ? 0 : fused->out_dtype;
  if (k == 0) {  // the empty sum
    if (fused != nullptr) {
      cudaError_t e = counted(launch_fused_k0(dtype == GEMM_TN_BF16, c, ldc, out_kind, m, n, fused->beta,
                                              fused->bias, fused->activation, dev->num_sms, stream));
      return e == cudaSuccess ? GEMM_TN_OK : fail_cuda(e, "fused epilogue (K = 0)");
    }
    cudaError_t e = cudaMemset2DAsync(c, static_cast<size_t>(ldc) * 2, 0, static_cast<size_t>(n) * 2,
                                      static_cast<size_t>(m), stream);
    return e == cudaSuccess ? GEMM_TN_OK : fail_cuda(e, "cudaMemset2DAsync");
  }
  const bool bf16 = dtype == GEMM_TN_BF16;

  int sk_resident[3];
  splitk_resident(dev, bf16, sk_resident);
  int cfg_id = choose_config(m, n, k, resident_clusters(dev, kCfg2CtaN256, bf16),
                             resident_clusters(dev, kCfg2CtaN256Mc, bf16), sk_resident);
  // multicast loads only from this GPU's own memory (also when forced)
  if (cfg_id == kCfg2CtaN256Mc && !multicast_source_ok(a, b)) cfg_id = kCfg2CtaN256;
  // the fused epilogue is built for the pair 256 x 256 and single-CTA 128 x 128 tiles
  if (fused != nullptr && cfg_id != kCfg1CtaN128) cfg_id = m <= 128 ? kCfg1CtaN128 : kCfg2CtaN256;
  // B stored [K, N] is built for 128- and 256-column tiles
  if (b_mn && cfg_id == kCfg1CtaN64) cfg_id = kCfg1CtaN128;
  // split-K: K cut over a cluster of `splits` CTAs per 128 x 128 tile (plain
  // K-major GEMM only; a forced split-K that cannot cut K runs whole tiles)
  int splits = 0;
  int decode = 0;   // rows of A per MMA of the decode kernel (0: not that kernel)
  if (cfg_id == kCfgDecodeSplitK) {
    decode = b_mn ? 0 : decode_rows(m);
    cfg_id = decode > 0 ? kCfgDecodeSplitK : kCfg1CtaSplitK;
  }
  if (cfg_id == kCfg1CtaSplitK || cfg_id == kCfgDecodeSplitK) {
    splits = resolve_splits(m, n, k, b_mn, dev->num_sms, sk_resident);
    if (splits < 2) {
      cfg_id = kCfg1CtaN128;
      decode = 0;
    }
  }
  const ConfigInfo& cfg = kConfigs[cfg_id];
  const int64_t num_m_tiles = (m + cfg.tile_m - 1) / cfg.tile_m;
  // columns per scheduled tile: a multicast cluster covers two pairs' tiles
  const int64_t cluster_n = static_cast<int64_t>(cfg.block_n) * cfg.cluster_pairs;
  const int64_t num_n_tiles = (n + cluster_n - 1) / cluster_n;
  const int64_t num_k_blocks = (k + kBlockK - 1) / kBlockK;
  const int64_t tiles = num_m_tiles * num_n_tiles;
  if (tiles > INT32_MAX) return fail(GEMM_TN_ERR_INVALID_VALUE, "too many output tiles");
  const int clusters = resident_clusters(dev, cfg_id, bf16);
  if (clusters <= 0) return fail(GEMM_TN_ERR_CUDA, "kernel cannot be resident on this device (occupancy query)");
  // The no-alloc path keeps to whole tiles: its fixed scratch is for repacks.
  WorkPlan plan = plan_work(tiles, num_k_blocks, clusters,
                            fixed_scratch == nullptr && splits == 0 ? stream_k_mode() : 0);
  int64_t split_begin = tiles;
  // split-capable kernels exist for the two CTA-pair configurations of the plain GEMM
  const bool can_split = !b_mn && fused == nullptr && (cfg_id == kCfg2CtaN256 || cfg_id == kCfg2CtaN256Mc);
  const int split = plan.sk_iters > 0 || !can_split ? 1 : tail_split(cfg, tiles, clusters, &split_begin, b_mn);
  if (split > 1) {
    const int64_t units = split_begin + (tiles - split_begin) * split;
    plan.workers = static_cast<int>(std::min<int64_t>(units, clusters));
  }
  // split-K: one cluster of `splits` CTAs per tile
  if (splits > 0 && tiles * splits > INT32_MAX) return fail(GEMM_TN_ERR_INVALID_VALUE, "too many output tiles");
  const int grid_ctas =
      splits > 0 ? static_cast<int>(tiles * splits) : plan.workers * cfg.cta_group * cfg.cluster_pairs;

  // Workspace: [repacked A][repacked B][stream-K partials][stream-K flags].
  // Operands the TMA cannot address directly are copied into padded rows.
  const bool repack_a = !tma_compatible(a, lda);
  const bool repack_b = !tma_compatible(b, ldb);
  const int64_t ld_pad = round_up(k, 8);
  // B rows: N rows of K elements, or (b_mn) K rows of N elements
  const int64_t b_rows_mem = b_mn ? k : n, b_cols_mem = b_mn ? n : k;
  const int64_t ldb_pad = round_up(b_cols_mem, 8);
  const size_t a_bytes = repack_a ? static_cast<size_t>(round_up(m * ld_pad * 2, 256)) : 0;
  const size_t b_bytes = repack_b ? static_cast<size_t>(round_up(b_rows_mem * ldb_pad * 2, 256)) : 0;
  const size_t partial_bytes =
      plan.sk_iters > 0 ? static_cast<size_t>(grid_ctas) * 128 * static_cast<size_t>(cfg.block_n) * 4 : 0;
  const size_t flag_bytes =
      plan.sk_iters > 0 ? static_cast<size_t>(grid_ctas) * gemm_tn_dev::kNumEpilogueWarps * sizeof(uint64_t) : 0;
  const size_t ws_bytes = a_bytes + b_bytes + partial_bytes + flag_bytes;
  void* workspace = nullptr;
  void* owned_workspace = nullptr;   // what this call allocated and must free
  cudaError_t e = cudaSuccess;
  if (ws_bytes > 0) {
    if (fixed_scratch != nullptr) {
      if (ws_bytes > fixed_scratch_bytes) {
        char buf[160];
        std::snprintf(buf, sizeof(buf),
                      "repack needs %zu bytes of scratch, more than the %zu-byte static scratch of the no-alloc path",
                      ws_bytes, fixed_scratch_bytes);
        return fail(GEMM_TN_ERR_INVALID_VALUE, buf);
      }
      workspace = fixed_scratch;
    } else {
      int dev_id = -1;
      cudaMemPool_t pool = nullptr;
      e = cudaGetDevice(&dev_id);
      if (e == cudaSuccess) e = dev_id >= 0 && dev_id < 64 ? workspace_pool(dev_id, &pool) : cudaErrorInvalidDevice;
      if (e != cudaSuccess) return fail_cuda(e, "workspace pool");
      e = cudaMallocFromPoolAsync(&workspace, ws_bytes, pool, stream);
      if (e != cudaSuccess) return fail_cuda(e, "cudaMallocFromPoolAsync (workspace)");
      owned_workspace = workspace;
    }
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const void* a_use = a;
  const void* b_use = b;
  int64_t lda_use = lda, ldb_use = ldb;
  if (repack_a || repack_b) {
    RepackRequest req[2] = {{a, lda, ws, ld_pad, repack_a ? m : 0, k},
                            {b, ldb, ws + a_bytes, ldb_pad, repack_b ? b_rows_mem : 0, b_cols_mem}};
    e = counted(launch_repack2(req, 2, dev->num_sms, stream));
    if (repack_a) {
      a_use = ws;
      lda_use = ld_pad;
    }
    if (repack_b) {
      b_use = ws + a_bytes;
      ldb_use = ldb_pad;
    }
  }
  if (e != cudaSuccess) {
    if (owned_workspace) cudaFreeAsync(owned_workspace, stream);
    return fail_cuda(e, "repack launch");
  }
  float* partials = partial_bytes ? reinterpret_cast<float*>(ws + a_bytes + b_bytes) : nullptr;
  uint64_t* flags = flag_bytes ? reinterpret_cast<uint64_t*>(ws + a_bytes + b_bytes + partial_bytes) : nullptr;

  alignas(64) gemm_tn_dev::GemmArgs args;
  std::memset(&args, 0, sizeof(args));
  // The split-K and decode kernels move two k-blocks per copy when K is a
  // multiple of 64 and every CTA of their clusters still gets at least one
  // pair; so do the 128 x 128 and 128 x 64 single-CTA tiles when every unit
  // of work covers all of K in order (no stream-K tail, tail split or rotated
  // K walk) and no fused epilogue is asked for (1024 x 2048 x 1024: 7.18 ->
  // 6.58 us per call replayed).
  const bool single_cta = cfg_id == kCfg1CtaN128 || cfg_id == kCfg1CtaN64;
  const bool main_pairs = single_cta && splits == 0 && fused == nullptr && !b_mn && k > 0 && k % 64 == 0 &&
                          plan.sk_iters == 0 && split == 1 && !k_rotation_on(num_m_tiles);
  const bool k_pairs = main_pairs || (splits > 0 && !b_mn && k % 64 == 0 && (k / 64 + 1) / 2 >= splits);
  if (k_pairs) {
    st = encode_kpair_map(&args.tmap_a, bf16, a_use, m, k, lda_use, decode > 0 ? decode : 128);
    if (st == GEMM_TN_OK)
      st = encode_kpair_map(&args.tmap_b, bf16, b_use, n, k, ldb_use, main_pairs ? cfg.b_rows : 128);
  } else {
    st = encode_matrix_map(&args.tmap_a, bf16, a_use, m, k, lda_use, kBlockK, decode > 0 ? decode : cfg.a_box_rows,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (k_pairs) {
    // B's map is set above
  } else if (st == GEMM_TN_OK && b_mn)   // [K, N]: 64 N x 64 K boxes
    st = encode_matrix_map(&args.tmap_b, bf16, b_use, k, n, ldb_use, 64, kBlockK, CU_TENSOR_MAP_SWIZZLE_128B);
  else if (st == GEMM_TN_OK)
    st = encode_matrix_map(&args.tmap_b, bf16, b_use, n, k, ldb_use, kBlockK, cfg.b_rows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == GEMM_TN_OK && split > 1 && !b_mn)
    st = encode_matrix_map(&args.tmap_b_split, bf16, b_use, n, k, ldb_use, kBlockK, cfg.b_rows / split,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  // C goes out through the TMA when its base and pitch allow; otherwise the
  // epilogue's predicated element stores handle any 2-byte-aligned layout.
  const bool c_tma = out_kind == 0 && tma_compatible(c, ldc) && !force_direct_epilogue();
  if (st == GEMM_TN_OK && c_tma)
    st = encode_matrix_map(&args.tmap_c, bf16, c, m, n, ldc, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (st != GEMM_TN_OK) {
    if (owned_workspace) cudaFreeAsync(owned_workspace, stream);
    return st;
  }
  args.c = c;
  args.ldc = ldc;
  args.c_tma_store = c_tma ? 1 : 0;
  args.m = static_cast<int32_t>(m);
  args.n = static_cast<int32_t>(n);
  args.k = static_cast<int32_t>(k);
  args.num_m_tiles = static_cast<int32_t>(num_m_tiles);
  args.num_n_tiles = static_cast<int32_t>(num_n_tiles);
  args.num_k_blocks = static_cast<int32_t>(num_k_blocks);
  args.num_tiles = static_cast<int32_t>(tiles);
  args.group_m = static_cast<int32_t>(std::min<int64_t>(group_rows(cfg), num_m_tiles));
  {
    // group_m <= num_m_tiles, so a group spans at most num_tiles (< 2^31) tiles
    const int64_t last_first_row = (num_m_tiles - 1) / args.group_m * args.group_m;
    args.div_group = make_fast_div(static_cast<int64_t>(args.group_m) * num_n_tiles);
    args.div_rows = make_fast_div(args.group_m);
    args.div_last_rows = make_fast_div(num_m_tiles - last_first_row);
    args.div_m_tiles = make_fast_div(num_m_tiles);
  }
  args.status = d_status;
  args.timeout_ns = watchdog_ns();
  args.drop_load_kb = drop_load_kb;
  args.dp_tiles = static_cast<int32_t>(plan.dp_tiles);
  args.num_workers = plan.workers;
  args.sk_iters = plan.sk_iters;
  args.sk_workers = plan.sk_workers;
  args.partials = partials;
  args.flags = flags;
  args.flag_epoch = flags != nullptr ? next_flag_epoch() : 0;
  args.split = split;
  args.split_log2 = split == 4 ? 2 : (split == 2 ? 1 : 0);
  args.split_begin = static_cast<int32_t>(split_begin);
  args.dp_units = static_cast<int32_t>(split_begin + (plan.dp_tiles - split_begin) * split);
  // one row of tiles: B streams from HBM once and A is re-read from L2
  args.k_rotate = k_rotation_on(num_m_tiles) ? 1 : 0;
  args.b_evict_first = args.k_rotate;
  if (fused != nullptr) {
    args.alpha = fused->alpha;
    args.beta = fused->beta;
    args.bias = fused->bias;
    args.activation = fused->activation;
    args.out_kind = out_kind;
  }

  if (decode > 0)
    e = counted(launch_gemm_decode(splits, decode, bf16, k_pairs, args, grid_ctas, stream));
  else if (splits > 0)
    e = counted(launch_gemm_splitk(splits, bf16, k_pairs, args, grid_ctas, stream));
  else if (fused != nullptr)
    e = counted(launch_gemm_fused(cfg_id, bf16, args, grid_ctas, stream));
  else if (b_mn)
    e = counted(launch_gemm_nn(cfg_id, bf16, args, grid_ctas, stream));
  else
    e = counted(cfg.cta_group == 2 ? launch_gemm_2cta(cfg_id, bf16, args, grid_ctas, stream)
                                   : launch_gemm_1cta(cfg_id, bf16, main_pairs, args, grid_ctas, stream));
  if (owned_workspace) {
    cudaError_t e2 = cudaFreeAsync(owned_workspace, stream);
    if (e == cudaSuccess) e = e2;
  }
  if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
  t_last_config = cfg_id;
  return GEMM_TN_OK;
}

// ---------------------------------------------------------------- no-alloc scratch
//
// Scratch for gemm_tn_ex_noalloc: file-scope device memory that every GPU
// loading this library holds until the process exits. Only the repack of a
// misaligned operand uses it. In host code `g_noalloc_scratch` names a host-side
// stand-in, not device memory, so its device address is looked up once per
// device (with that device current) and cached.
__device__ __align__(256) uint8_t g_noalloc_scratch[GEMM_TN_NOALLOC_SCRATCH_BYTES];

// The address is cached per device together with the context it was looked
// up in: a different current context on that device (a context the caller
// created, or the primary context after cudaDeviceReset) holds its own copy of
// the array, so the lookup is repeated when the context changes.
struct ScratchAddr {
  CUcontext ctx = nullptr;
  void* addr = nullptr;
};
std::mutex g_scratch_mutex;
ScratchAddr g_scratch_addr[64];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
std::once_flag g_ctx_once;

// The current driver context (nullptr when it cannot be read).
CUcontext current_context() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    } else {
      cudaGetLastError();
    }
  });
  CUcontext ctx = nullptr;
  if (g_ctx_get_current == nullptr || g_ctx_get_current(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

int noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return fail(GEMM_TN_ERR_UNSUPPORTED_DEVICE, "no current CUDA device");
  }
  // cudaGetDevice does not create the primary context; the lookup below does,
  // so a call with no context yet takes the lookup path and caches the new one
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchAddr& slot = g_scratch_addr[dev];
  if (slot.addr == nullptr || ctx == nullptr || slot.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return fail_cuda(e, "cudaGetSymbolAddress (no-alloc scratch)");
    slot.addr = p;
    slot.ctx = current_context();
  }
  *out = slot.addr;
  return GEMM_TN_OK;
}

// ---------------------------------------------------------------- host-buffer path
//
// Per-device resources of gemm_tn_host, created on its first call on a device
// and kept until the process exits: two copy streams (host-to-device and
// device-to-host), the events that chain copies and GEMMs, and a memory pool
// that keeps the staging memory between calls instead of returning it to the
// system at every synchronisation.
struct HostPath {
  static constexpr int kMaxChunks = 16;
  bool ready = false;
  std::mutex mutex;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev_start = nullptr, ev_b = nullptr, ev_done = nullptr;
  cudaEvent_t ev_a[kMaxChunks] = {}, ev_c[kMaxChunks] = {};
  cudaMemPool_t pool = nullptr;
};

std::mutex g_host_path_mutex;
HostPath g_host_path[64];

int host_path(HostPath** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return fail(GEMM_TN_ERR_UNSUPPORTED_DEVICE, "no current CUDA device");
  }
  std::lock_guard<std::mutex> lock(g_host_path_mutex);
  HostPath& hp = g_host_path[dev];
  if (!hp.ready) {
    cudaError_t e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking);
    const unsigned flags = cudaEventDisableTiming;
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.ev_start, flags);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.ev_b, flags);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.ev_done, flags);
    for (int i = 0; i < HostPath::kMaxChunks && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&hp.ev_a[i], flags);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.ev_c[i], flags);
    }
    if (e == cudaSuccess) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.handleTypes = cudaMemHandleTypeNone;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      e = cudaMemPoolCreate(&hp.pool, &props);
    }
    if (e == cudaSuccess) {
      uint64_t keep = UINT64_MAX;
      e = cudaMemPoolSetAttribute(hp.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    }
    if (e != cudaSuccess) return fail_cuda(e, "host-path set-up");
    hp.ready = true;
  }
  *out = &hp;
  return GEMM_TN_OK;
}

}  // namespace

const ConfigInfo& config_info(int id) { return kConfigs[id]; }

bool dependent_launch_enabled() {
  static const bool on = [] {
    const char* s = std::getenv("GEMM_TN_PDL");
    return s == nullptr || std::strcmp(s, "0") != 0;
  }();
  return on;
}

}  // namespace gemm_tn_impl

using namespace gemm_tn_impl;

extern "C" {

int gemm_tn(int dtype, int64_t m, int64_t n, int64_t k, const void* a, const void* b, void* c,
            gemm_tn_stream_t stream) {
  return run_gemm(dtype, m, n, k, a, k, b, k, c, n, nullptr, reinterpret_cast<cudaStream_t>(stream), -1);
}

int gemm_tn_ex(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda, const void* b, int64_t ldb,
               void* c, int64_t ldc, int* d_status, gemm_tn_stream_t stream) {
  return run_gemm(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status, reinterpret_cast<cudaStream_t>(stream),
                  test_drop_load_kb());
}

int gemm_tn_fused(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda, const void* b, int64_t ldb,
                  void* c, int64_t ldc, const gemm_tn_epilogue* epilogue, int* d_status, gemm_tn_stream_t stream) {
  t_last_cuda_error = 0;
  t_last_message[0] = '\0';
  if (epilogue == nullptr) return fail(GEMM_TN_ERR_INVALID_VALUE, "epilogue is NULL");
  if (epilogue->activation < GEMM_TN_ACT_NONE || epilogue->activation > GEMM_TN_ACT_GELU)
    return fail(GEMM_TN_ERR_INVALID_VALUE, "unknown activation");
  if (epilogue->out_dtype != GEMM_TN_OUT_INPUT && epilogue->out_dtype != GEMM_TN_OUT_F32 &&
      epilogue->out_dtype != GEMM_TN_OUT_E4M3)
    return fail(GEMM_TN_ERR_INVALID_VALUE, "unknown output dtype");
  if (epilogue->bias != nullptr && reinterpret_cast<uintptr_t>(epilogue->bias) % 4)
    return fail(GEMM_TN_ERR_MISALIGNED, "bias is not 4-byte aligned");
  // C's alignment and its overlap with A and B are checked for C's own
  // element size by run_gemm's validation
  return run_gemm(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status, reinterpret_cast<cudaStream_t>(stream),
                  test_drop_load_kb(), nullptr, 0, false, epilogue);
}

int gemm_nn(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda, const void* b, int64_t ldb,
            void* c, int64_t ldc, int* d_status, gemm_tn_stream_t stream) {
  return run_gemm(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status, reinterpret_cast<cudaStream_t>(stream),
                  test_drop_load_kb(), nullptr, 0, /*b_mn=*/true);
}

int gemm_tn_ex_noalloc(int dtype, int64_t m, int64_t n, int64_t k, const void* a, int64_t lda, const void* b,
                       int64_t ldb, void* c, int64_t ldc, int* d_status, gemm_tn_stream_t stream) {
  t_last_cuda_error = 0;
  t_last_message[0] = '\0';
  int st = validate(dtype, m, n, k, a, lda, b, ldb, c, ldc);
  if (st != GEMM_TN_OK || m == 0 || n == 0) return st;
  DeviceFacts* facts = nullptr;
  st = current_device(&facts);
  if (st != GEMM_TN_OK) return st;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != GEMM_TN_OK) return st;
  return run_gemm(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status, reinterpret_cast<cudaStream_t>(stream), -1,
                  scratch, GEMM_TN_NOALLOC_SCRATCH_BYTES);
}

int gemm_tn_host(int dtype, int64_t m, int64_t n, int64_t k, const void* a_host, const void* b_host, void* c_host,
                 gemm_tn_stream_t stream_handle) {
  t_last_cuda_error = 0;
  t_last_message[0] = '\0';
  int st = validate(dtype, m, n, k, a_host, k, b_host, k, c_host, n);
  if (st != GEMM_TN_OK || m == 0 || n == 0) return st;
  DeviceFacts* facts = nullptr;
  st = current_device(&facts);
  if (st != GEMM_TN_OK) return st;
  HostPath* hp = nullptr;
  st = host_path(&hp);
  if (st != GEMM_TN_OK) return st;
  std::lock_guard<std::mutex> serial(hp->mutex);   // one host-buffer call per device at a time
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);

  // Device staging with 16-byte row pitches: no repack, TMA-store epilogue.
  const int64_t ldk = round_up(std::max<int64_t>(k, 1), 8), ldn = round_up(n, 8);
  const size_t a_bytes = static_cast<size_t>(round_up(m * ldk * 2, 256));
  const size_t b_bytes = static_cast<size_t>(round_up(n * ldk * 2, 256));
  const size_t c_bytes = static_cast<size_t>(round_up(m * ldn * 2, 256));
  uint8_t* dev_buf = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dev_buf), a_bytes + b_bytes + c_bytes + 256,
                                          hp->pool, stream);
  if (e != cudaSuccess) return fail_cuda(e, "cudaMallocFromPoolAsync (host-path staging)");
  uint16_t* d_a = reinterpret_cast<uint16_t*>(dev_buf);
  uint16_t* d_b = reinterpret_cast<uint16_t*>(dev_buf + a_bytes);
  uint16_t* d_c = reinterpret_cast<uint16_t*>(dev_buf + a_bytes + b_bytes);
  int* d_status = reinterpret_cast<int*>(dev_buf + a_bytes + b_bytes + c_bytes);

  // Rows of A (and C) go in chunks of whole 256-row tiles, about 16 MB of A
  // each, so the copies in both directions overlap the GEMMs of earlier chunks.
  const int64_t a_host_bytes = m * k * 2;
  int64_t chunks = std::min<int64_t>(HostPath::kMaxChunks, std::max<int64_t>(1, a_host_bytes / (16ll << 20)));
  int64_t rows_per = round_up((m + chunks - 1) / chunks, 256);
  chunks = (m + rows_per - 1) / rows_per;

  int rc = GEMM_TN_OK;
  auto check = [&](cudaError_t err, const char* what) {
    if (rc == GEMM_TN_OK && err != cudaSuccess) rc = fail_cuda(err, what);
  };
  check(cudaMemsetAsync(d_status, 0, sizeof(int), stream), "cudaMemsetAsync (status)");
  check(cudaEventRecord(hp->ev_start, stream), "cudaEventRecord");
  check(cudaStreamWaitEvent(hp->h2d, hp->ev_start, 0), "cudaStreamWaitEvent");
  if (k > 0) {
    check(cudaMemcpy2DAsync(d_b, ldk * 2, b_host, k * 2, k * 2, n, cudaMemcpyHostToDevice, hp->h2d), "copy B");
  }
  check(cudaEventRecord(hp->ev_b, hp->h2d), "cudaEventRecord");
  check(cudaStreamWaitEvent(stream, hp->ev_b, 0), "cudaStreamWaitEvent");
  for (int64_t i = 0; i < chunks && rc == GEMM_TN_OK; ++i) {
    const int64_t r0 = i * rows_per, rows = std::min(rows_per, m - r0);
    if (k > 0) {
      check(cudaMemcpy2DAsync(d_a + r0 * ldk, ldk * 2, static_cast<const uint8_t*>(a_host) + r0 * k * 2, k * 2,
                              k * 2, rows, cudaMemcpyHostToDevice, hp->h2d),
            "copy A");
    }
    check(cudaEventRecord(hp->ev_a[i], hp->h2d), "cudaEventRecord");
    check(cudaStreamWaitEvent(stream, hp->ev_a[i], 0), "cudaStreamWaitEvent");
    if (rc != GEMM_TN_OK) break;
    const int gst = run_gemm(dtype, rows, n, k, d_a + r0 * ldk, ldk, d_b, ldk, d_c + r0 * ldn, ldn, d_status, stream,
                             -1);
    if (gst != GEMM_TN_OK) {
      rc = gst;
      break;
    }
    check(cudaEventRecord(hp->ev_c[i], stream), "cudaEventRecord");
    check(cudaStreamWaitEvent(hp->d2h, hp->ev_c[i], 0), "cudaStreamWaitEvent");
    check(cudaMemcpy2DAsync(static_cast<uint8_t*>(c_host) + r0 * n * 2, n * 2, d_c + r0 * ldn, ldn * 2, n * 2, rows,
                            cudaMemcpyDeviceToHost, hp->d2h),
          "copy C");
  }
  int h_status = 0;
  check(cudaMemcpyAsync(&h_status, d_status, sizeof(int), cudaMemcpyDeviceToHost, hp->d2h), "copy status");
  // the staging buffer goes back to the pool only after every copy is done
  cudaEventRecord(hp->ev_done, hp->d2h);
  cudaStreamWaitEvent(stream, hp->ev_done, 0);
  cudaError_t ef = cudaFreeAsync(dev_buf, stream);
  cudaError_t es = cudaStreamSynchronize(stream);
  check(ef, "cudaFreeAsync");
  check(es, "cudaStreamSynchronize");
  if (rc == GEMM_TN_OK && h_status != 0) rc = fail(h_status, "device watchdog expired");
  return rc;
}

int flash_attn_fwd(int dtype, int64_t batch, int64_t seq, int64_t heads, int64_t head_dim, const void* q,
                   const void* k, const void* v, void* o, float softmax_scale, int causal, int* d_status,
                   gemm_tn_stream_t stream) {
  t_last_cuda_error = 0;
  t_last_message[0] = '\0';
  if (dtype != GEMM_TN_F16 && dtype != GEMM_TN_BF16) return fail(GEMM_TN_ERR_UNSUPPORTED_DTYPE, "dtype");
  if (batch < 0 || seq < 0 || heads < 0) return fail(GEMM_TN_ERR_INVALID_VALUE, "negative size");
  if (head_dim != 64 && head_dim != 128) return fail(GEMM_TN_ERR_INVALID_VALUE, "head_dim must be 64 or 128");
  if (!(softmax_scale >= 0.0f) || !std::isfinite(softmax_scale))
    return fail(GEMM_TN_ERR_INVALID_VALUE, "softmax_scale must be finite and non-negative");
  if (batch == 0 || seq == 0 || heads == 0) return GEMM_TN_OK;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return fail(GEMM_TN_ERR_INVALID_VALUE, "NULL pointer");
  // one batch [seq, heads, dim] must stay under 2^39 bytes (tensor-map strides),
  // and the grid and the kernel's indices under 2^31
  const int64_t q_tiles = (seq + flash_attn_rows_per_cta() - 1) / flash_attn_rows_per_cta();   // CTAs per head
  if (seq > kMaxDim || heads > kMaxDim || batch > kMaxDim || heads * head_dim > (int64_t{1} << 30) ||
      seq * heads * head_dim > (int64_t{1} << 38) || batch * heads > kMaxDim || q_tiles * batch * heads > kMaxDim)
    return fail(GEMM_TN_ERR_INVALID_VALUE, "sizes past the limits");
  for (const void* p : {static_cast<const void*>(q), k, v, static_cast<const void*>(o)})
    if (reinterpret_cast<uintptr_t>(p) % 16) return fail(GEMM_TN_ERR_MISALIGNED, "pointer not 16-byte aligned");
  const uintptr_t bytes = static_cast<uintptr_t>(batch * seq * heads * head_dim * 2);
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(o);
  for (const void* p : {q, k, v}) {
    const uintptr_t p0 = reinterpret_cast<uintptr_t>(p);
    if (ranges_overlap(o0, o0 + bytes, p0, p0 + bytes)) return fail(GEMM_TN_ERR_INVALID_VALUE, "O overlaps an input");
  }
  DeviceFacts* facts = nullptr;
  int st = current_device(&facts);
  if (st != GEMM_TN_OK) return st;

  const bool bf16 = dtype == GEMM_TN_BF16;
  gemm_tn_dev::FlashArgs args{};
  if ((st = encode_bshd_map(&args.tmap_q, bf16, q, batch, seq, heads, head_dim)) != GEMM_TN_OK) return st;
  if ((st = encode_bshd_map(&args.tmap_k, bf16, k, batch, seq, heads, head_dim)) != GEMM_TN_OK) return st;
  if ((st = encode_bshd_map(&args.tmap_v, bf16, v, batch, seq, heads, head_dim)) != GEMM_TN_OK) return st;
  const double scale = softmax_scale > 0.0f ? static_cast<double>(softmax_scale) : 1.0 / std::sqrt(static_cast<double>(head_dim));
  args.o = o;
  args.batch = static_cast<int>(batch);
  args.seq = static_cast<int>(seq);
  args.heads = static_cast<int>(heads);
  args.num_q_tiles = static_cast<int>(q_tiles);
  args.scale_log2 = static_cast<float>(scale * 1.4426950408889634);   // log2(e)
  args.causal = causal != 0 ? 1 : 0;
  args.status = d_status;
  args.timeout_ns = watchdog_ns();
  args.drop_load_block = test_drop_load_kb();
  // heads whose K and V (2 * seq * dim * 2 bytes each) fit in ~48 MB of L2
  // together run their query tiles interleaved
  const int64_t kv_bytes = 2 * seq * head_dim * 2;
  args.head_group = static_cast<int>(std::min<int64_t>(batch * heads, std::max<int64_t>(1, (48ll << 20) / kv_bytes)));
  const unsigned grid = static_cast<unsigned>(q_tiles * batch * heads);
  const cudaError_t e = counted(launch_flash_attn(static_cast<int>(head_dim), bf16, args, grid,
                                                  reinterpret_cast<cudaStream_t>(stream)));
  if (e != cudaSuccess) return fail_cuda(e, "flash attention launch");
  return GEMM_TN_OK;
}

namespace {

// What the selection sees for a dtype on the current device: resident CTA
// pairs, 4-CTA clusters, split-K clusters of 2, 4, 8 CTAs, and SMs; GB300's
// when there is no usable device.
void selection_facts(int dtype, int* pairs, int* quads, int sk[3], int* sms) {
  *pairs = 76;
  *quads = 36;
  *sms = 152;
  for (int i = 0; i < 3; ++i) sk[i] = kGb300SplitKResidentDefault[i];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  DeviceFacts* facts = nullptr;
  if (current_device(&facts) != GEMM_TN_OK) return;
  const bool bf16 = dtype == GEMM_TN_BF16;
  const int p = resident_clusters(facts, kCfg2CtaN256, bf16);
  const int q = resident_clusters(facts, kCfg2CtaN256Mc, bf16);
  if (p > 0 && q > 0) {
    *pairs = p;
    *quads = q;
  }
  splitk_resident(facts, bf16, sk);
  *sms = facts->num_sms;
}

bool selectable(int dtype, int64_t m, int64_t n, int64_t k) {
  return (dtype == GEMM_TN_F16 || dtype == GEMM_TN_BF16) && m > 0 && n > 0 && k > 0 && m <= kMaxDim &&
         n <= kMaxDim && k <= kMaxDim;
}

}  // namespace

int gemm_tn_select_config(int dtype, int64_t m, int64_t n, int64_t k) {
  if (!selectable(dtype, m, n, k)) return -1;
  int pairs, quads, sms, sk[3];
  selection_facts(dtype, &pairs, &quads, sk, &sms);
  return choose_config(m, n, k, pairs, quads, sk);
}

int gemm_tn_select_splits(int dtype, int64_t m, int64_t n, int64_t k) {
  if (!selectable(dtype, m, n, k)) return 0;
  int pairs, quads, sms, sk[3];
  selection_facts(dtype, &pairs, &quads, sk, &sms);
  const int cfg = choose_config(m, n, k, pairs, quads, sk);
  if (cfg != kCfg1CtaSplitK && cfg != kCfgDecodeSplitK) return 0;
  return resolve_splits(m, n, k, false, sms, sk);
}

int gemm_tn_last_config(void) { return t_last_config; }

void* gemm_tn_workspace_pool(void) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  cudaMemPool_t pool = nullptr;
  return workspace_pool(dev, &pool) == cudaSuccess ? static_cast<void*>(pool) : nullptr;
}

int gemm_tn_trim_workspace(void) {
  t_last_cuda_error = 0;
  t_last_message[0] = '\0';
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return fail(GEMM_TN_ERR_UNSUPPORTED_DEVICE, "no current CUDA device");
  }
  cudaMemPool_t pool = nullptr;
  e = workspace_pool(dev, &pool);
  if (e == cudaSuccess) e = cudaMemPoolTrimTo(pool, 0);
  return e == cudaSuccess ? GEMM_TN_OK : fail_cuda(e, "cudaMemPoolTrimTo (workspace pool)");
}

int gemm_tn_multicast_allowed(const void* a, const void* b) { return multicast_source_ok(a, b) ? 1 : 0; }

int gemm_tn_num_configs(void) { return kNumConfigs; }

const char* gemm_tn_config_name(int config) {
  if (config < 0 || config >= kNumConfigs) return "invalid";
  return kConfigs[config].name;
}

const char* gemm_tn_status_string(int status) {
  switch (status) {
    case GEMM_TN_OK: return "GEMM_TN_OK";
    case GEMM_TN_ERR_INVALID_VALUE: return "GEMM_TN_ERR_INVALID_VALUE";
    case GEMM_TN_ERR_UNSUPPORTED_DTYPE: return "GEMM_TN_ERR_UNSUPPORTED_DTYPE";
    case GEMM_TN_ERR_MISALIGNED: return "GEMM_TN_ERR_MISALIGNED";
    case GEMM_TN_ERR_UNSUPPORTED_DEVICE: return "GEMM_TN_ERR_UNSUPPORTED_DEVICE";
    case GEMM_TN_ERR_CUDA: return "GEMM_TN_ERR_CUDA";
    case GEMM_TN_ERR_TIMEOUT: return "GEMM_TN_ERR_TIMEOUT";
    default: return "GEMM_TN_ERR_UNKNOWN";
  }
}

int gemm_tn_last_cuda_error(void) { return t_last_cuda_error; }

const char* gemm_tn_last_error_message(void) { return t_last_message; }

int gemm_tn_version(void) { return kAbiVersion; }

uint64_t gemm_tn_launch_count(void) { return g_launch_count.load(std::memory_order_relaxed); }

}  // extern "C"
