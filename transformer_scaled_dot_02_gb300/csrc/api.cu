// The C ABI of libsdpa (declared in include/sdpa.h): argument checks, tensor
// maps for the TMA, and the launches of the attention and projection kernels.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "sdpa.h"

namespace {

using sdpa::GemmParams;
using sdpa::GemmProblem;
using sdpa::SdpaF32Params;
using sdpa::SdpaTcParams;

// Error word the kernels raise bits in (bounded waits that gave up).
__device__ unsigned g_device_status;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool probed = false;
  bool supported = false;
  unsigned* status = nullptr;  // device address of g_device_status
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

// Kernel pins set by sdpa_set_kernel_choice; 0 = choose by shape.
std::atomic<int> g_pin_attention{0};       // 1 = one-tile kernel, 2 = two-tile kernel
std::atomic<int> g_pin_one_tile_keys{0};   // 32 | 64
std::atomic<int> g_pin_gemm_bn{0};         // 128 | 256

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// Checks that the current device is a GB300-class (sm_103) GPU and returns its
// status-word address.  The first call on a device does the probing.
sdpa_status current_device(unsigned** status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SDPA_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return SDPA_ERR_UNSUPPORTED_DEVICE;
    }
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) {
        cudaGetLastError();
        return SDPA_ERR_CUDA;
      }
      st.status = static_cast<unsigned*>(addr);
    }
    st.probed = true;
  }
  if (!st.supported) return SDPA_ERR_UNSUPPORTED_DEVICE;
  *status = st.status;
  return SDPA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Key spans up to these lengths use the one-tile kernel (d <= 128); longer
// walks use the two-tile kernel.  Measured on GB300 (b = 4, 16 * 8192 / n
// heads, d = 16 to 128): the kernels are within 1-3 % at 3072 keys; at 512
// keys the one-tile kernel leads by up to 40 %, at 8192 keys the two-tile
// kernel by up to 13 % (d = 16 and 32, causal).  A restricted window keeps
// every query tile's walk short, and the one-tile kernel leads up to r = 4096
// (within 2 % there).
constexpr long long kOneTileMaxKeys = 3072;
constexpr long long kOneTileShortKeys = 2048;   // d = 64: 32-key tiles up to this span
constexpr long long kOneTileMaxKeysWindowed = 4352;   // r up to 4096
constexpr long long kKvBytesOneGroup = 32ll << 20;    // K + V of all heads: one work group

// 4-D bf16 map over (d, n, h, b) with the given element strides of n, h, b;
// boxes of min(d, 64) x 128, swizzled at the row width, zero fill outside.
bool make_map_4d(CUtensorMap* map, const void* base, int d, int n, int h, int b,
                 long long stride_n, long long stride_h, long long stride_b, int box_rows = 128) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n > 0 ? n : 1),
                              static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(b)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(stride_n) * 2,
                                 static_cast<cuuint64_t>(stride_h) * 2,
                                 static_cast<cuuint64_t>(stride_b) * 2};
  // boxes of min(d, 64) columns: rows of 128, 64 or 32 bytes, swizzled at that width
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(d < 64 ? d : 64),
                             static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle swz = d >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                         : (d == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                    : CU_TENSOR_MAP_SWIZZLE_32B);
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 map over the backward's dQ accumulator [bh][n_q][d]: boxes of
// min(32, d) columns x box_rows rows, unswizzled, for the kernel's tensor
// reduce-adds; rows past n_q are clipped by the copy engine.
bool make_map_dq(CUtensorMap* map, const float* base, int d, int n_q, int bh, int box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n_q > 0 ? n_q : 1),
                              static_cast<cuuint64_t>(bh)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(n_q > 0 ? n_q : 1) * d * 4};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(d < 32 ? d : 32),
                             static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 map over a row-major [rows, cols] matrix: box (64 cols, box_rows).
bool make_map_2d(CUtensorMap* map, const void* base, int rows, int cols, int box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared argument rules of the attention entry points (host-only checks).
sdpa_status check_attention_args(const void* q, const void* k, const void* v, const void* out,
                                 int b, int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                                 const int32_t* kv_lengths, float scale) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return SDPA_ERR_INVALID_ARG;
  if (b < 1 || h < 1 || n_q < 0 || n_k < 0 || d_k < 1 || d_v < 1) return SDPA_ERR_INVALID_ARG;
  if (mask_kind < 0 || mask_kind > (SDPA_MASK_CAUSAL | SDPA_MASK_PADDING))
    return SDPA_ERR_INVALID_ARG;
  if ((mask_kind & SDPA_MASK_CAUSAL) && n_q != n_k) return SDPA_ERR_INVALID_ARG;
  if ((mask_kind & SDPA_MASK_PADDING) &&
      (kv_lengths == nullptr || (reinterpret_cast<uintptr_t>(kv_lengths) & 3u) != 0))
    return SDPA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return SDPA_ERR_INVALID_ARG;
  if (n_q >= sdpa::kWindowUnbounded || n_k >= sdpa::kWindowUnbounded) return SDPA_ERR_UNSUPPORTED;
  // Sizes must stay addressable by the TMA (dimension <= 2^32, strides < 2^40 bytes).
  const long long elems_q = 1ll * b * h * n_q * (d_k > d_v ? d_k : d_v);
  const long long elems_k = 1ll * b * h * n_k * (d_k > d_v ? d_k : d_v);
  if (elems_q > (1ll << 38) || elems_k > (1ll << 38)) return SDPA_ERR_UNSUPPORTED;
  return SDPA_OK;
}

// head sizes the tensor-core attention kernel is built for
bool tc_head_size(int d) {
  return d == 16 || d == 32 || d == 64 || d == 128 || d == 256 || d == 512;
}

// (d_k, d_v) pairs the tensor-core attention is built for: equal sizes, or
// the smaller keys of Table 3's rows (B) against 64-wide values.
bool tc_head_sizes(int d_k, int d_v) {
  if (d_k == d_v) return tc_head_size(d_k);
  return d_v == 64 && (d_k == 16 || d_k == 32);
}

// Head shapes the backward supports: every equal size of Table 3 and its
// rows (B), where the keys are smaller than the values.
bool bwd_head_sizes(int d_k, int d_v) {
  if (d_k == d_v) return tc_head_size(d_k);
  return d_v == 64 && (d_k == 16 || d_k == 32);
}

float effective_scale(float scale, int d_k) {
  return scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k)));
}

// Kernel choice for tensor-core attention.  sdpa_set_kernel_choice pins it
// (tests use this to cover both kernels on the same shapes); otherwise it is
// picked by shape, from the measurements on GB300 given with the thresholds
// above.
// Keys one 128-row query tile can see at most.
long long key_span(int n_k, int win_left, int win_right) {
  return std::min<long long>(n_k, 1ll * win_left + win_right + 128);
}

bool use_one_tile_kernel(int d, int n_k, int win_left, int win_right) {
  if (d > 128) return true;
  const int pin = g_pin_attention.load(std::memory_order_relaxed);
  if (pin == 1) return true;
  if (pin == 2) return false;
  const long long span = key_span(n_k, win_left, win_right);
  const bool windowed = win_left != sdpa::kWindowUnbounded || win_right != sdpa::kWindowUnbounded;
  return span <= (windowed ? kOneTileMaxKeysWindowed : kOneTileMaxKeys);
}

// Key tile of the one-tile kernel: 32 below d = 64, 64 above.  At d = 64,
// 32-key tiles need 128 tensor-memory columns, so four CTAs share an SM
// instead of two; that pays when the walk is short and the grid holds at
// least two waves of two-CTA slots (measured on GB300: 6-17 % faster on
// 1024-key walks and restricted windows, 15 % on b32 h16 256 x 384; 22 %
// slower on b32 h8 n128, 2 % on 3072-key walks).  sdpa_set_kernel_choice
// pins it at d = 64.
int one_tile_key_tile(int d, long long span, long long ctas) {
  if (d < 64) return 32;
  if (d > 64) return 64;
  const int pin = g_pin_one_tile_keys.load(std::memory_order_relaxed);
  if (pin == 32 || pin == 64) return pin;
  return (span <= kOneTileShortKeys && ctas >= 4ll * sdpa::device_sm_count()) ? 32 : 64;
}

// Element strides of a 4-D (d, n, h, b) tensor along n, h and b.
struct Strides {
  long long n, h, b;
};
Strides bhsd(int h, int n, int d) { return {d, 1ll * n * d, 1ll * h * n * d}; }
Strides bshd(int h, int n, int d) { return {1ll * h * d, d, 1ll * n * h * d}; }

// Launches the tensor-core attention over tensors with arbitrary (n, h, b)
// element strides (BHSD for sdpa_forward, BSHD inside mha_forward).  The
// launch carries a programmatic dependency on the previous kernel in the
// stream: the CTAs may start and set up early, and read or write global
// memory only after griddep_wait(), so any predecessor stays safe.
sdpa_status launch_attention_tc(const void* q, const void* k, const void* v, void* out, int b,
                                int h, int n_q, int n_k, int d_k, int d_v, Strides sq, Strides sk,
                                Strides sv, Strides so, int mask_kind, const int32_t* kv_lengths,
                                float scale, unsigned* status, cudaStream_t stream,
                                int win_left = sdpa::kWindowUnbounded,
                                int win_right = sdpa::kWindowUnbounded, float* lse = nullptr,
                                bool pdl = true) {
  SdpaTcParams p;
  p.pdl = pdl ? 1 : 0;
  // The one-tile kernel (one 128-row query tile per CTA, 32- or 64-key tiles;
  // two or four CTAs per SM at d <= 128) takes wide heads and the short key
  // walks where the two-tile kernel's longer per-CTA chain would leave SMs
  // idle.  Unequal key and value sizes take the two-tile one.
  const bool one_tile = d_k == d_v && use_one_tile_kernel(d_k, n_k, win_left, win_right);
  const int kv_rows =
      one_tile ? one_tile_key_tile(d_k, key_span(n_k, win_left, win_right),
                                   1ll * ((n_q + 127) / 128) * b * h)
               : 128;
  if (one_tile && !sdpa::one_tile_supports(d_k, kv_rows)) return SDPA_ERR_UNSUPPORTED;
  if (!make_map_4d(&p.tm_q, q, d_k, n_q, h, b, sq.n, sq.h, sq.b) ||
      !make_map_4d(&p.tm_k, k, d_k, n_k, h, b, sk.n, sk.h, sk.b, kv_rows) ||
      !make_map_4d(&p.tm_v, v, d_v, n_k, h, b, sv.n, sv.h, sv.b, kv_rows) ||
      !make_map_4d(&p.tm_o, out, d_v, n_q, h, b, so.n, so.h, so.b))
    return SDPA_ERR_CUDA;
  p.kv_lengths = (mask_kind & SDPA_MASK_PADDING) ? kv_lengths : nullptr;
  p.status = status;
  p.b = b;
  p.h = h;
  p.n_q = n_q;
  p.n_k = n_k;
  p.mask_kind = mask_kind;
  p.num_q_blocks = one_tile ? (n_q + 127) / 128 : (n_q + 255) / 256;
  p.scale_log2 = effective_scale(scale, d_k) * 1.4426950408889634f;
  p.win_left = win_left;
  p.win_right = win_right;
  p.lse = lse;
  // One-tile kernel: heads in groups of 8 keep their K and V in L2 on long
  // sequences; when the K and V of all heads fit in a quarter of L2 the
  // whole grid is one group, so the longest causal query tiles of every
  // head start first and the short ones fill in behind them.
  p.head_group = 8;
  if (one_tile) {
    const long long kv_bytes = 2ll * b * h * n_k * (d_k + d_v);
    const int units = b * h * (d_k == 512 ? 2 : 1);
    if (kv_bytes <= kKvBytesOneGroup) p.head_group = units;
  }
  const cudaError_t err = one_tile ? sdpa::launch_sdpa_one_tile(p, d_k, kv_rows, stream)
                                   : sdpa::launch_sdpa_tc(p, d_k, d_v, stream);
  return err == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

bool fill_gemm_problem(GemmProblem* pr, const void* x, const void* w, void* y, int m, int n,
                       int k) {
  pr->m = m;
  pr->n = n;
  pr->k = k;
  return make_map_2d(&pr->tm_a, x, m, k, sdpa::kGemmBlockM) && make_map_2d(&pr->tm_b, w, k, n, 64) &&
         make_map_2d(&pr->tm_c, y, m, n, sdpa::kGemmBlockM);
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Streams and events of the host-buffer pipeline (sdpa_forward_host), made
// once per device on its first call and kept for the process.
struct HostPipeline {
  bool ready = false;
  cudaStream_t copy_in = nullptr, compute = nullptr, copy_out = nullptr;
  cudaEvent_t start = nullptr, in_done = nullptr, cmp_done = nullptr, end = nullptr;
  std::mutex mutex;   // one enqueue at a time: the events are re-recorded per chunk
};
HostPipeline g_pipelines[kMaxDevices];

sdpa_status host_pipeline(HostPipeline** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SDPA_ERR_UNSUPPORTED_DEVICE;
  }
  HostPipeline& hp = g_pipelines[dev];
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!hp.ready) {
    const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&hp.copy_in, sf) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.compute, sf) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.copy_out, sf) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.start, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.in_done, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.cmp_done, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.end, ef) != cudaSuccess) {
      cudaGetLastError();
      return SDPA_ERR_CUDA;
    }
    hp.ready = true;
  }
  *out = &hp;
  return SDPA_OK;
}

// Decode: enough splits for about kDecodeWaves waves of the shape's resident
// CTAs; the workspace is sized for the most any shape can take.
int decode_target_ctas(int resident) {
  return sdpa::kDecodeWaves * resident * sdpa::device_sm_count();
}

}  // namespace

namespace sdpa {
int gemm_bn_pin() { return g_pin_gemm_bn.load(std::memory_order_relaxed); }
}  // namespace sdpa

extern "C" {

sdpa_status sdpa_set_kernel_choice(int attention_kernel, int one_tile_keys, int gemm_bn) {
  if (attention_kernel < 0 || attention_kernel > 2) return SDPA_ERR_INVALID_ARG;
  if (one_tile_keys != 0 && one_tile_keys != 32 && one_tile_keys != 64)
    return SDPA_ERR_INVALID_ARG;
  if (gemm_bn != 0 && gemm_bn != 128 && gemm_bn != 256) return SDPA_ERR_INVALID_ARG;
  g_pin_attention.store(attention_kernel, std::memory_order_relaxed);
  g_pin_one_tile_keys.store(one_tile_keys, std::memory_order_relaxed);
  g_pin_gemm_bn.store(gemm_bn, std::memory_order_relaxed);
  return SDPA_OK;
}

sdpa_status sdpa_forward(const void* q, const void* k, const void* v, void* out, int b, int h,
                         int n_q, int n_k, int d_k, int d_v, int mask_kind,
                         const int32_t* kv_lengths, float scale, void* stream) {
  sdpa_status st = check_attention_args(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind,
                                        kv_lengths, scale);
  if (st != SDPA_OK) return st;
  if (!tc_head_sizes(d_k, d_v)) return SDPA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  st = current_device(&status);
  if (st != SDPA_OK) return st;
  if (n_q == 0) return SDPA_OK;
  return launch_attention_tc(q, k, v, out, b, h, n_q, n_k, d_k, d_v, bhsd(h, n_q, d_k),
                             bhsd(h, n_k, d_k), bhsd(h, n_k, d_v), bhsd(h, n_q, d_v), mask_kind,
                             kv_lengths, scale, status, static_cast<cudaStream_t>(stream));
}

sdpa_status sdpa_forward_restricted(const void* q, const void* k, const void* v, void* out,
                                    int b, int h, int n_q, int n_k, int d_k, int d_v,
                                    int mask_kind, const int32_t* kv_lengths, int r, float scale,
                                    void* stream) {
  sdpa_status st = check_attention_args(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind,
                                        kv_lengths, scale);
  if (st != SDPA_OK) return st;
  if (r < 1) return SDPA_ERR_INVALID_ARG;
  if (!tc_head_sizes(d_k, d_v)) return SDPA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  st = current_device(&status);
  if (st != SDPA_OK) return st;
  if (n_q == 0) return SDPA_OK;
  // a neighbourhood of r positions: floor((r-1)/2) before i, floor(r/2) after
  const int left = (r - 1) / 2, right = r / 2;
  return launch_attention_tc(q, k, v, out, b, h, n_q, n_k, d_k, d_v, bhsd(h, n_q, d_k),
                             bhsd(h, n_k, d_k), bhsd(h, n_k, d_v), bhsd(h, n_q, d_v), mask_kind,
                             kv_lengths, scale, status, static_cast<cudaStream_t>(stream), left,
                             right);
}

sdpa_status sdpa_forward_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                             int b, int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                             const int32_t* kv_lengths, int r, float scale, void* stream) {
  sdpa_status st = check_attention_args(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind,
                                        kv_lengths, scale);
  if (st != SDPA_OK) return st;
  if (lse == nullptr || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 || r < 0)
    return SDPA_ERR_INVALID_ARG;
  if (!tc_head_sizes(d_k, d_v)) return SDPA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  st = current_device(&status);
  if (st != SDPA_OK) return st;
  if (n_q == 0) return SDPA_OK;
  const int left = r > 0 ? (r - 1) / 2 : sdpa::kWindowUnbounded;
  const int right = r > 0 ? r / 2 : sdpa::kWindowUnbounded;
  return launch_attention_tc(q, k, v, out, b, h, n_q, n_k, d_k, d_v, bhsd(h, n_q, d_k),
                             bhsd(h, n_k, d_k), bhsd(h, n_k, d_v), bhsd(h, n_q, d_v), mask_kind,
                             kv_lengths, scale, status, static_cast<cudaStream_t>(stream), left,
                             right, lse);
}

size_t sdpa_backward_workspace_size(int b, int h, int n_q, int d) {
  if (b < 1 || h < 1 || n_q < 0 || d < 1) return 0;
  const size_t rows_pad = static_cast<size_t>(b) * h * ((n_q + 127) / 128 * 128);
  return 2 * round256(rows_pad * 4) + round256(static_cast<size_t>(b) * h * n_q * d * 4);
}

sdpa_status sdpa_backward(const void* q, const void* k, const void* v, const void* out,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv,
                          void* workspace, size_t ws_bytes, int b, int h, int n_q, int n_k,
                          int d_k, int d_v, int mask_kind, const int32_t* kv_lengths, int r,
                          float scale, void* stream) {
  sdpa_status st = check_attention_args(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind,
                                        kv_lengths, scale);
  if (st != SDPA_OK) return st;
  if (dout == nullptr || lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 || r < 0)
    return SDPA_ERR_INVALID_ARG;
  if (!bwd_head_sizes(d_k, d_v)) return SDPA_ERR_UNSUPPORTED;
  const size_t need = sdpa_backward_workspace_size(b, h, n_q, d_k);
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < need) return SDPA_ERR_WORKSPACE;
  unsigned* status = nullptr;
  st = current_device(&status);
  if (st != SDPA_OK) return st;
  if (n_q == 0 && n_k == 0) return SDPA_OK;
  const int n_q_pad = (n_q + 127) / 128 * 128;
  const size_t rows_pad = static_cast<size_t>(b) * h * n_q_pad;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* neg_lse2 = reinterpret_cast<float*>(ws);
  float* neg_dvec = reinterpret_cast<float*>(ws + round256(rows_pad * 4));
  float* dq_acc = reinterpret_cast<float*>(ws + 2 * round256(rows_pad * 4));
  sdpa::SdpaBwdParams bp;
  const long long dk_ = d_k, dv_ = d_v;
  // the backward steps through the queries 64 (32 for 512-wide heads) at a
  // time, against key tiles of 128 (64) rows
  const int q_rows = sdpa::bwd_query_step(d_k), key_rows = sdpa::bwd_key_tile(d_k);
  if (!make_map_4d(&bp.tm_q, q, d_k, n_q, h, b, dk_, n_q * dk_, h * n_q * dk_, q_rows) ||
      !make_map_4d(&bp.tm_k, k, d_k, n_k, h, b, dk_, n_k * dk_, h * n_k * dk_, key_rows) ||
      !make_map_4d(&bp.tm_v, v, d_v, n_k, h, b, dv_, n_k * dv_, h * n_k * dv_, key_rows) ||
      !make_map_4d(&bp.tm_do, dout, d_v, n_q, h, b, dv_, n_q * dv_, h * n_q * dv_, q_rows))
    return SDPA_ERR_CUDA;
  // heads wider than 128 reduce dQ 32 query rows at a time
  if (!make_map_dq(&bp.tm_dq, dq_acc, d_k, n_q, b * h, d_k > 128 ? 32 : 64)) return SDPA_ERR_CUDA;
  bp.neg_lse2 = neg_lse2;
  bp.neg_dvec = neg_dvec;
  bp.dq_acc = dq_acc;
  bp.dk = static_cast<uint16_t*>(dk);
  bp.dv = static_cast<uint16_t*>(dv);
  bp.kv_lengths = (mask_kind & SDPA_MASK_PADDING) ? kv_lengths : nullptr;
  bp.status = status;
  bp.b = b;
  bp.h = h;
  bp.n_q = n_q;
  bp.n_k = n_k;
  bp.n_q_pad = n_q_pad;
  bp.mask_kind = mask_kind;
  bp.num_kv_tiles = (n_k + key_rows - 1) / key_rows;
  const float sc = effective_scale(scale, d_k);
  bp.scale_log2 = sc * 1.4426950408889634f;
  bp.scale = sc;
  bp.win_left = r > 0 ? (r - 1) / 2 : sdpa::kWindowUnbounded;
  bp.win_right = r > 0 ? r / 2 : sdpa::kWindowUnbounded;
  sdpa::SdpaBwdPrepParams pp;
  pp.out = static_cast<const uint16_t*>(out);
  pp.dout = static_cast<const uint16_t*>(dout);
  pp.lse = lse;
  pp.neg_lse2 = neg_lse2;
  pp.neg_dvec = neg_dvec;
  pp.dq_acc = dq_acc;
  pp.dq = static_cast<uint16_t*>(dq);
  pp.b = b;
  pp.h = h;
  pp.n_q = n_q;
  pp.n_q_pad = n_q_pad;
  pp.scale = sc;
  return sdpa::launch_sdpa_bwd(bp, pp, d_k, d_v, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SDPA_OK
             : SDPA_ERR_CUDA;
}

sdpa_status sdpa_forward_host(const void* q_host, const void* k_host, const void* v_host,
                              void* out_host, void* q_dev, void* k_dev, void* v_dev, void* out_dev,
                              int b, int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                              const int32_t* kv_lengths, float scale, int heads_per_chunk,
                              void* stream) {
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr || out_host == nullptr)
    return SDPA_ERR_INVALID_ARG;
  sdpa_status st = check_attention_args(q_dev, k_dev, v_dev, out_dev, b, h, n_q, n_k, d_k, d_v,
                                        mask_kind, kv_lengths, scale);
  if (st != SDPA_OK) return st;
  if (heads_per_chunk < 0) return SDPA_ERR_INVALID_ARG;
  if (!tc_head_sizes(d_k, d_v)) return SDPA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  st = current_device(&status);
  if (st != SDPA_OK) return st;
  if (n_q == 0) return SDPA_OK;
  HostPipeline* hp = nullptr;
  st = host_pipeline(&hp);
  if (st != SDPA_OK) return st;
  std::lock_guard<std::mutex> lock(hp->mutex);
  cudaStream_t main = static_cast<cudaStream_t>(stream);
  const int hc = (heads_per_chunk == 0 || heads_per_chunk > h) ? h : heads_per_chunk;
  // bytes of one (batch, head) slice of each tensor; a chunk of heads of one
  // batch entry is contiguous in BHSD
  const size_t qb = static_cast<size_t>(n_q) * d_k * 2, kb = static_cast<size_t>(n_k) * d_k * 2;
  const size_t vb = static_cast<size_t>(n_k) * d_v * 2, ob = static_cast<size_t>(n_q) * d_v * 2;
  auto bad = [](cudaError_t e) {
    if (e == cudaSuccess) return false;
    cudaGetLastError();
    return true;
  };
  // everything after the work already queued on the caller's stream
  if (bad(cudaEventRecord(hp->start, main)) ||
      bad(cudaStreamWaitEvent(hp->copy_in, hp->start, 0)) ||
      bad(cudaStreamWaitEvent(hp->compute, hp->start, 0)) ||
      bad(cudaStreamWaitEvent(hp->copy_out, hp->start, 0)))
    return SDPA_ERR_CUDA;
  for (int bi = 0; bi < b; ++bi) {
    for (int h0 = 0; h0 < h; h0 += hc) {
      const int nh = h - h0 < hc ? h - h0 : hc;
      const size_t slice = static_cast<size_t>(bi) * h + h0;
      auto at = [&](const void* base, size_t bytes) {
        return static_cast<const uint8_t*>(base) + slice * bytes;
      };
      auto at_mut = [&](void* base, size_t bytes) { return static_cast<uint8_t*>(base) + slice * bytes; };
      if (bad(cudaMemcpyAsync(at_mut(q_dev, qb), at(q_host, qb), nh * qb, cudaMemcpyHostToDevice,
                              hp->copy_in)) ||
          bad(cudaMemcpyAsync(at_mut(k_dev, kb), at(k_host, kb), nh * kb, cudaMemcpyHostToDevice,
                              hp->copy_in)) ||
          bad(cudaMemcpyAsync(at_mut(v_dev, vb), at(v_host, vb), nh * vb, cudaMemcpyHostToDevice,
                              hp->copy_in)) ||
          bad(cudaEventRecord(hp->in_done, hp->copy_in)) ||
          bad(cudaStreamWaitEvent(hp->compute, hp->in_done, 0)))
        return SDPA_ERR_CUDA;
      st = launch_attention_tc(at(q_dev, qb), at(k_dev, kb), at(v_dev, vb), at_mut(out_dev, ob), 1,
                               nh, n_q, n_k, d_k, d_v, bhsd(nh, n_q, d_k), bhsd(nh, n_k, d_k),
                               bhsd(nh, n_k, d_v), bhsd(nh, n_q, d_v), mask_kind,
                               kv_lengths != nullptr ? kv_lengths + bi : nullptr, scale, status,
                               hp->compute, sdpa::kWindowUnbounded, sdpa::kWindowUnbounded,
                               nullptr, /*pdl=*/false);
      if (st != SDPA_OK) return st;
      if (bad(cudaEventRecord(hp->cmp_done, hp->compute)) ||
          bad(cudaStreamWaitEvent(hp->copy_out, hp->cmp_done, 0)) ||
          bad(cudaMemcpyAsync(at_mut(out_host, ob), at(out_dev, ob), nh * ob,
                              cudaMemcpyDeviceToHost, hp->copy_out)))
        return SDPA_ERR_CUDA;
    }
  }
  // the caller's stream continues after the last copy back
  if (bad(cudaEventRecord(hp->end, hp->copy_out)) || bad(cudaStreamWaitEvent(main, hp->end, 0)))
    return SDPA_ERR_CUDA;
  return SDPA_OK;
}

sdpa_status sdpa_forward_f32(const void* q, const void* k, const void* v, void* out, int b, int h,
                             int n_q, int n_k, int d_k, int d_v, int mask_kind,
                             const int32_t* kv_lengths, float scale, void* stream) {
  sdpa_status st = check_attention_args(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind,
                                        kv_lengths, scale);
  if (st != SDPA_OK) return st;
  if (d_k > 128 || d_v > 128 || 1ll * b * h > 65535) return SDPA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  st = current_device(&status);
  if (st != SDPA_OK) return st;
  if (n_q == 0) return SDPA_OK;
  SdpaF32Params p;
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.out = static_cast<float*>(out);
  p.kv_lengths = (mask_kind & SDPA_MASK_PADDING) ? kv_lengths : nullptr;
  p.b = b;
  p.h = h;
  p.n_q = n_q;
  p.n_k = n_k;
  p.d_k = d_k;
  p.d_v = d_v;
  p.mask_kind = mask_kind;
  p.scale = effective_scale(scale, d_k);
  return sdpa::launch_sdpa_f32(p, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SDPA_OK
             : SDPA_ERR_CUDA;
}

size_t sdpa_decode_workspace_size(int b, int h, int n_q, int n_k, int d_v) {
  if (b < 1 || h < 1 || n_q < 1 || n_k < 0 || d_v < 1) return 0;
  const int splits =
      sdpa::decode_splits(b, h, n_k, decode_target_ctas(sdpa::kDecodeMaxResident));
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(b) * h * n_q;
  return round256(static_cast<size_t>(splits) * rows * d_v * 4) +
         round256(static_cast<size_t>(splits) * rows * 2 * 4);
}

sdpa_status sdpa_decode(const void* q, const void* k, const void* v, void* out, void* workspace,
                        size_t ws_bytes, int b, int h, int n_q, int n_k, int d_k, int d_v,
                        const int32_t* kv_lengths, float scale, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return SDPA_ERR_INVALID_ARG;
  if (b < 1 || h < 1 || n_q < 1 || n_k < 0 || d_k < 1 || d_v < 1) return SDPA_ERR_INVALID_ARG;
  if (kv_lengths != nullptr && (reinterpret_cast<uintptr_t>(kv_lengths) & 3u) != 0)
    return SDPA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return SDPA_ERR_INVALID_ARG;
  if (!sdpa::decode_supports(d_k, d_v) || n_q > sdpa::kDecodeMaxQueries ||
      1ll * b * h > 65535 || n_k >= sdpa::kWindowUnbounded ||
      1ll * b * h * n_k * (d_k > d_v ? d_k : d_v) > (1ll << 38))
    return SDPA_ERR_UNSUPPORTED;
  const size_t need = sdpa_decode_workspace_size(b, h, n_q, n_k, d_v);
  if (need > 0 && (workspace == nullptr || !aligned16(workspace) || ws_bytes < need))
    return SDPA_ERR_WORKSPACE;
  unsigned* status = nullptr;
  sdpa_status st = current_device(&status);
  if (st != SDPA_OK) return st;
  sdpa::DecodeParams p;
  const int tk = sdpa::decode_keys_per_tile(d_k);
  if (!make_map_4d(&p.tm_k, k, d_k, n_k, h, b, d_k, 1ll * n_k * d_k, 1ll * h * n_k * d_k, tk) ||
      !make_map_4d(&p.tm_v, v, d_v, n_k, h, b, d_v, 1ll * n_k * d_v, 1ll * h * n_k * d_v, tk))
    return SDPA_ERR_CUDA;
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  p.kv_lengths = kv_lengths;
  p.status = status;
  p.b = b;
  p.h = h;
  p.n_q = n_q;
  p.n_k = n_k;
  // never more splits than the workspace was sized for (resident <= the maximum)
  p.splits = sdpa::decode_splits(b, h, n_k,
                                 decode_target_ctas(sdpa::decode_resident_ctas(d_k, d_v)));
  const int per = (n_k + p.splits - 1) / p.splits;
  p.keys_per_split = (per + tk - 1) / tk * tk;
  const size_t rows = static_cast<size_t>(b) * h * n_q;
  p.part_o = p.splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.part_ml = p.splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                      round256(static_cast<size_t>(p.splits) *
                                                               rows * d_v * 4))
                           : nullptr;
  p.scale_log2 = effective_scale(scale, d_k) * 1.4426950408889634f;
  return sdpa::launch_sdpa_decode(p, d_k, d_v, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SDPA_OK
             : SDPA_ERR_CUDA;
}

size_t mha_workspace_size(int b, int n_q, int n_k, int h, int d_k, int d_v) {
  if (b < 0 || n_q < 0 || n_k < 0 || h < 0 || d_k < 0 || d_v < 0) return 0;
  const size_t bq = static_cast<size_t>(b) * n_q, bk = static_cast<size_t>(b) * n_k;
  return round256(bq * h * d_k * 2) + round256(bk * h * d_k * 2) + round256(bk * h * d_v * 2) +
         round256(bq * h * d_v * 2);
}

sdpa_status mha_forward(const void* xq, const void* xkv, const void* wq, const void* wk,
                        const void* wv, const void* wo, void* y, void* workspace, size_t ws_bytes,
                        int b, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                        int mask_kind, const int32_t* kv_lengths, float scale, void* stream) {
  if (xq == nullptr || xkv == nullptr || wq == nullptr || wk == nullptr || wv == nullptr ||
      wo == nullptr || y == nullptr)
    return SDPA_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(xkv) || !aligned16(wq) || !aligned16(wk) || !aligned16(wv) ||
      !aligned16(wo) || !aligned16(y))
    return SDPA_ERR_INVALID_ARG;
  if (b < 1 || h < 1 || n_q < 0 || n_k < 0 || d_model < 1 || d_k < 1 || d_v < 1)
    return SDPA_ERR_INVALID_ARG;
  if (mask_kind < 0 || mask_kind > (SDPA_MASK_CAUSAL | SDPA_MASK_PADDING))
    return SDPA_ERR_INVALID_ARG;
  if ((mask_kind & SDPA_MASK_CAUSAL) && n_q != n_k) return SDPA_ERR_INVALID_ARG;
  if ((mask_kind & SDPA_MASK_PADDING) &&
      (kv_lengths == nullptr || (reinterpret_cast<uintptr_t>(kv_lengths) & 3u) != 0))
    return SDPA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return SDPA_ERR_INVALID_ARG;
  if (!tc_head_sizes(d_k, d_v) || d_model % 8 != 0) return SDPA_ERR_UNSUPPORTED;
  if (1ll * b * (n_q > n_k ? n_q : n_k) > (1ll << 30) || 1ll * h * (d_k > d_v ? d_k : d_v) > 65536)
    return SDPA_ERR_UNSUPPORTED;
  const size_t need = mha_workspace_size(b, n_q, n_k, h, d_k, d_v);
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < need) return SDPA_ERR_WORKSPACE;
  unsigned* status = nullptr;
  sdpa_status st = current_device(&status);
  if (st != SDPA_OK) return st;
  if (n_q == 0) return SDPA_OK;

  const size_t bq = static_cast<size_t>(b) * n_q, bk = static_cast<size_t>(b) * n_k;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qp = ws;
  void* kp = ws + round256(bq * h * d_k * 2);
  void* vp = static_cast<uint8_t*>(kp) + round256(bk * h * d_k * 2);
  void* op = static_cast<uint8_t*>(vp) + round256(bk * h * d_v * 2);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int m_q = static_cast<int>(bq), m_k = static_cast<int>(bk);
  const int hd = h * d_k, hv = h * d_v;

  // Q = X_q W^Q, K = X_kv W^K, V = X_kv W^V in one launch; outputs [b*n, h*d]
  // row-major, which is the per-head layout [b, n, h, d] the attention reads.
  GemmParams gp;
  gp.status = status;
  gp.num_problems = 0;
  gp.pdl = 1;   // the GEMM touches global memory only after griddep_wait()
  if (!fill_gemm_problem(&gp.prob[gp.num_problems++], xq, wq, qp, m_q, hd, d_model))
    return SDPA_ERR_CUDA;
  if (m_k > 0) {
    if (!fill_gemm_problem(&gp.prob[gp.num_problems++], xkv, wk, kp, m_k, hd, d_model) ||
        !fill_gemm_problem(&gp.prob[gp.num_problems++], xkv, wv, vp, m_k, hv, d_model))
      return SDPA_ERR_CUDA;
  }
  if (sdpa::launch_gemm_tc(gp, m_q > m_k ? m_q : m_k, hd > hv ? hd : hv, s) != cudaSuccess)
    return SDPA_ERR_CUDA;

  // Heads: strides of [b, n, h, d]; the output lands in Concat order.
  // The attention and the W^O product each launch with a programmatic
  // dependency on the kernel before them (as every attention launch does):
  // their CTAs start, allocate and set up while that kernel's last CTAs
  // finish, then wait for its results before reading anything.
  st = launch_attention_tc(qp, kp, vp, op, b, h, n_q, n_k, d_k, d_v, bshd(h, n_q, d_k),
                           bshd(h, n_k, d_k), bshd(h, n_k, d_v), bshd(h, n_q, d_v), mask_kind,
                           kv_lengths, scale, status, s, sdpa::kWindowUnbounded,
                           sdpa::kWindowUnbounded, nullptr, true);
  if (st != SDPA_OK) return st;

  // Y = Concat(heads) W^O
  GemmParams go;
  go.status = status;
  go.num_problems = 1;
  go.pdl = 1;
  if (!fill_gemm_problem(&go.prob[0], op, wo, y, m_q, d_model, h * d_v)) return SDPA_ERR_CUDA;
  return sdpa::launch_gemm_tc(go, m_q, d_model, s) == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

sdpa_status linear_forward(const void* x, const void* w, void* y, int m, int n, int k,
                           void* stream) {
  if (x == nullptr || w == nullptr || y == nullptr) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return SDPA_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || k < 1) return SDPA_ERR_INVALID_ARG;
  if (n % 8 != 0 || k % 8 != 0) return SDPA_ERR_UNSUPPORTED;
  if (m > (1 << 30)) return SDPA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  sdpa_status st = current_device(&status);
  if (st != SDPA_OK) return st;
  GemmParams gp;
  gp.status = status;
  gp.num_problems = 1;
  gp.pdl = 1;
  if (!fill_gemm_problem(&gp.prob[0], x, w, y, m, n, k)) return SDPA_ERR_CUDA;
  return sdpa::launch_gemm_tc(gp, m, n, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SDPA_OK
             : SDPA_ERR_CUDA;
}

sdpa_status sdpa_device_check(void) {
  unsigned* status = nullptr;
  sdpa_status st = current_device(&status);
  if (st != SDPA_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return SDPA_ERR_CUDA;
  }
  unsigned word = 0;
  const unsigned zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_device_status, sizeof(word)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess) {
    cudaGetLastError();
    return SDPA_ERR_CUDA;
  }
  return (word & sdpa::kStatusTimeout) ? SDPA_ERR_DEVICE_TIMEOUT : SDPA_OK;
}

const char* sdpa_status_string(sdpa_status status) {
  switch (status) {
    case SDPA_OK: return "SDPA_OK";
    case SDPA_ERR_INVALID_ARG: return "SDPA_ERR_INVALID_ARG";
    case SDPA_ERR_UNSUPPORTED: return "SDPA_ERR_UNSUPPORTED";
    case SDPA_ERR_UNSUPPORTED_DEVICE: return "SDPA_ERR_UNSUPPORTED_DEVICE";
    case SDPA_ERR_WORKSPACE: return "SDPA_ERR_WORKSPACE";
    case SDPA_ERR_CUDA: return "SDPA_ERR_CUDA";
    case SDPA_ERR_DEVICE_TIMEOUT: return "SDPA_ERR_DEVICE_TIMEOUT";
  }
  return "SDPA_ERR_UNKNOWN";
}

}  // extern "C"
