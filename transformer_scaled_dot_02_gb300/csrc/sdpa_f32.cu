// Scaled dot-product attention in fp32 on the CUDA cores ("Attention Is All
// You Need", section 3.2.1, Eq. (1), with the masks of section 3.2.3).
//
// For small fp32 problems and any head size 1..128.  Each warp owns
// kRowsPerWarp query rows and streams 32-key tiles of K and V through shared
// memory: lane j scores key j of the tile, the tile maximum and the sum of the
// exponentials are combined across the warp with shuffles (online softmax),
// and lane c accumulates output columns c, c+32, c+64, c+96.  Exponentials use
// the accurate expf (this file is built without fast-math), so the result
// carries fp32 rounding only.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;
constexpr int kKeyTile = 32;
constexpr int kMaxD = 128;
constexpr int kPad = kMaxD + 1;   // odd stride: lane j reads row j conflict-free

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Copies rows [0, rows) of a row-major [*, d] fp32 matrix (rows at and past
// `valid` read as 0) into a shared tile [rows][kPad].  With d a multiple of 4
// every thread issues all its 16-byte loads before any store, so their
// latencies overlap instead of adding up; other d take one float at a time.
template <int kRows>
__device__ __forceinline__ void load_tile(float (*dst)[kPad], const float* src, int valid, int d) {
  if ((d & 3) == 0) {
    constexpr int kPerThread = kRows * (kMaxD / 4) / (kWarps * 32);
    const int vpr = d / 4;   // 16-byte pieces per row
    float4 buf[kPerThread];
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const int idx = threadIdx.x + i * kWarps * 32;
      const int r = idx / vpr, c4 = idx % vpr;
      buf[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < kRows && r < valid)
        buf[i] = *reinterpret_cast<const float4*>(src + static_cast<long long>(r) * d + c4 * 4);
    }
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const int idx = threadIdx.x + i * kWarps * 32;
      const int r = idx / vpr, c4 = idx % vpr;
      if (r < kRows) {
        dst[r][c4 * 4 + 0] = buf[i].x;
        dst[r][c4 * 4 + 1] = buf[i].y;
        dst[r][c4 * 4 + 2] = buf[i].z;
        dst[r][c4 * 4 + 3] = buf[i].w;
      }
    }
  } else {
    for (int idx = threadIdx.x; idx < kRows * d; idx += kWarps * 32) {
      const int r = idx / d, c = idx % d;
      dst[r][c] = r < valid ? src[static_cast<long long>(r) * d + c] : 0.f;
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32)
sdpa_fwd_f32_simt(const SdpaF32Params p) {
  __shared__ float q_s[kRowsPerCta][kPad];
  __shared__ float k_s[kKeyTile][kPad];
  __shared__ float v_s[kKeyTile][kPad];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int bi = bh / p.h;
  const int row0 = blockIdx.x * kRowsPerCta;
  const float* q = p.q + static_cast<long long>(bh) * p.n_q * p.d_k;
  const float* k = p.k + static_cast<long long>(bh) * p.n_k * p.d_k;
  const float* v = p.v + static_cast<long long>(bh) * p.n_k * p.d_v;
  float* out = p.out + static_cast<long long>(bh) * p.n_q * p.d_v;

  const bool causal = (p.mask_kind & 1) != 0;
  // the next kernel may launch now; this grid's inputs may come from the
  // previous kernel in the stream, so wait for it before reading them
  griddep_launch_dependents();
  griddep_wait();
  int kv_len = p.n_k;
  if ((p.mask_kind & 2) && p.kv_lengths != nullptr) {
    kv_len = p.kv_lengths[bi];
    kv_len = kv_len < 0 ? 0 : (kv_len > p.n_k ? p.n_k : kv_len);
  }
  // Keys past the last visible one of the CTA's last row are never needed.
  int key_end = kv_len;
  if (causal) key_end = min(key_end, row0 + kRowsPerCta);

  load_tile<kRowsPerCta>(q_s, q + static_cast<long long>(row0) * p.d_k, p.n_q - row0, p.d_k);

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kMaxD / 32];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxD / 32; ++c) acc[r][c] = 0.f;
  }

  for (int key0 = 0; key0 < key_end; key0 += kKeyTile) {
    __syncthreads();  // previous tile fully consumed (and q_s written)
    load_tile<kKeyTile>(k_s, k + static_cast<long long>(key0) * p.d_k, p.n_k - key0, p.d_k);
    load_tile<kKeyTile>(v_s, v + static_cast<long long>(key0) * p.d_v, p.n_k - key0, p.d_v);
    __syncthreads();

#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int rl = warp * kRowsPerWarp + r;
      const int row = row0 + rl;
      const int key = key0 + lane;
      // score of key `key` for this row (lane-parallel over keys)
      float dot = 0.f;
      for (int c = 0; c < p.d_k; ++c) dot = fmaf(q_s[rl][c], k_s[lane][c], dot);
      const bool visible = key < kv_len && !(causal && key > row);
      const float s = visible ? dot * p.scale : -INFINITY;
      const float m_new = fmaxf(m[r], warp_max(s));
      // m_new == -inf: nothing visible yet in this row; keep everything at 0.
      const float alpha = (m_new == -INFINITY) ? 1.f : expf(m[r] - m_new);
      const float pj = (m_new == -INFINITY || !visible) ? 0.f : expf(s - m_new);
      l[r] = l[r] * alpha + warp_sum(pj);
      m[r] = m_new;
#pragma unroll
      for (int cc = 0; cc < kMaxD / 32; ++cc) acc[r][cc] *= alpha;
      for (int j = 0; j < kKeyTile; ++j) {
        const float w = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
        for (int cc = 0; cc < kMaxD / 32; ++cc) {
          const int c = cc * 32 + lane;
          if (c < p.d_v) acc[r][cc] = fmaf(w, v_s[j][c], acc[r][cc]);
        }
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int row = row0 + warp * kRowsPerWarp + r;
    if (row >= p.n_q) continue;
    const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
#pragma unroll
    for (int cc = 0; cc < kMaxD / 32; ++cc) {
      const int c = cc * 32 + lane;
      if (c < p.d_v) out[static_cast<long long>(row) * p.d_v + c] = acc[r][cc] * inv;
    }
  }
}

}  // namespace

cudaError_t launch_sdpa_f32(const SdpaF32Params& p, cudaStream_t stream) {
  const long long bh = static_cast<long long>(p.b) * p.h;
  if (bh == 0 || p.n_q == 0) return cudaSuccess;
  if (bh > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid((p.n_q + kRowsPerCta - 1) / kRowsPerCta, static_cast<unsigned>(bh));
  // a programmatic dependency on the previous kernel: the kernel reads
  // global memory only after griddep_wait()
  return launch_kernel(sdpa_fwd_f32_simt, grid, dim3(kWarps * 32), 0, stream, true, p);
}

}  // namespace sdpa
