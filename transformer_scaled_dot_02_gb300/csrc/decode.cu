// One autoregressive decoding step ("Attention Is All You Need", section 3.1:
// the decoder produces one symbol at a time): n_q <= 8 new queries per
// (batch, head) attend to a cached K/V of length len_b, query i seeing keys
// j <= len_b - n_q + i.  Eq. (1) with the causal rule of section 3.2.3.
//
// The step reads every cached key and value once and does 2 d FLOP per key
// and query, so it is bound by HBM bandwidth, not by the tensor cores.  It
// runs on the CUDA cores and splits each sequence's cache across CTAs so the
// whole GPU streams it:
//   sdpa_decode_split   grid (splits, b*h), 4 warps.  A warp walks groups of 8
//                       keys of its CTA's key range; lane l holds columns
//                       [l*d/32, (l+1)*d/32) of the 8 K and V rows (coalesced
//                       row loads).  Partial dot products are summed with a
//                       butterfly reduce-scatter (9 shuffles for 8 keys) that
//                       leaves key (lane >> 2) & 7 on each lane; the group's
//                       max and exponential sum are shuffle reductions; an
//                       online softmax updates (m, l, O) per query.  The 4
//                       warps merge through shared memory, then the CTA writes
//                       either the final output (one split) or its partial
//                       (m, l, O) to the workspace.
//   sdpa_decode_combine merges the splits' partials: O = sum_s O_s 2^(m_s-M) /
//                       sum_s l_s 2^(m_s-M), M = max_s m_s.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int kDecThreads = 128;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kGroup = 8;  // keys per warp step

// Lane `lane`'s d/32 columns of one bf16 row, widened to fp32.
template <int D>
__device__ __forceinline__ void load_row(const uint16_t* row, int lane, float (&x)[D / 32]) {
  if constexpr (D == 128) {
    const uint2 u = *reinterpret_cast<const uint2*>(row + 4 * lane);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(row + 2 * lane);
    x[0] = __uint_as_float(u << 16);
    x[1] = __uint_as_float(u & 0xffff0000u);
  }
}

// Sums 8 per-lane partial values over the warp; lane l returns the total of
// value (l >> 2) & 7.  Butterfly: halve the values kept at each of the lane
// bits 4, 3, 2, then add over lane bits 0 and 1.
__device__ __forceinline__ float reduce_scatter8(const float (&v)[8], int lane) {
  float a[4], b2[2];
  const bool h4 = (lane >> 4) & 1, h3 = (lane >> 3) & 1, h2 = (lane >> 2) & 1;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float keep = h4 ? v[4 + t] : v[t];
    const float send = h4 ? v[t] : v[4 + t];
    a[t] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const float keep = h3 ? a[2 + t] : a[t];
    const float send = h3 ? a[t] : a[2 + t];
    b2[t] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float keep = h2 ? b2[1] : b2[0];
  const float send = h2 ? b2[0] : b2[1];
  float s = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  return s;
}

// max / sum over the 8 keys held by lane groups (lane bits 2..4)
__device__ __forceinline__ float group_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
}
__device__ __forceinline__ float group_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  return x + __shfl_xor_sync(0xffffffffu, x, 16);
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
  return static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xffffu);
}

template <int D, int MAXQ>
__global__ void __launch_bounds__(kDecThreads) sdpa_decode_split(const DecodeParams p) {
  griddep_launch_dependents();   // the combine kernel may launch now
  constexpr int C = D / 32;
  __shared__ float sm_m[kDecWarps][MAXQ], sm_l[kDecWarps][MAXQ];
  __shared__ float sm_o[kDecWarps][MAXQ][D];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int bh = blockIdx.y;
  const int bi = bh / p.h;
  int len = p.n_k;
  if (p.kv_lengths != nullptr) {
    len = p.kv_lengths[bi];
    len = len < 0 ? 0 : (len > p.n_k ? p.n_k : len);
  }
  const int c0 = split * p.keys_per_split;
  const int c1 = min(c0 + p.keys_per_split, len);
  const uint16_t* kb = p.k + static_cast<long long>(bh) * p.n_k * D;
  const uint16_t* vb = p.v + static_cast<long long>(bh) * p.n_k * D;

  // queries, pre-scaled so that scores come out in log2 units
  float qv[MAXQ][C];
#pragma unroll
  for (int i = 0; i < MAXQ; ++i) {
    if (i < p.n_q) {
      load_row<D>(p.q + (static_cast<long long>(bh) * p.n_q + i) * D, lane, qv[i]);
#pragma unroll
      for (int c = 0; c < C; ++c) qv[i][c] *= p.scale_log2;
    } else {
#pragma unroll
      for (int c = 0; c < C; ++c) qv[i][c] = 0.f;
    }
  }
  float m[MAXQ], l[MAXQ], o[MAXQ][C];
#pragma unroll
  for (int i = 0; i < MAXQ; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) o[i][c] = 0.f;
  }

  for (int g0 = c0 + warp * kGroup; g0 < c1; g0 += kDecWarps * kGroup) {
    float kf[kGroup][C], vf[kGroup][C];
#pragma unroll
    for (int kk = 0; kk < kGroup; ++kk) {
      const int j = g0 + kk;
      if (j < c1) {
        load_row<D>(kb + static_cast<long long>(j) * D, lane, kf[kk]);
        load_row<D>(vb + static_cast<long long>(j) * D, lane, vf[kk]);
      } else {
#pragma unroll
        for (int c = 0; c < C; ++c) kf[kk][c] = vf[kk][c] = 0.f;
      }
    }
    const int my_key = g0 + ((lane >> 2) & 7);
#pragma unroll
    for (int i = 0; i < MAXQ; ++i) {
      if (i >= p.n_q) break;
      float part[kGroup];
#pragma unroll
      for (int kk = 0; kk < kGroup; ++kk) {
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) acc = fmaf(qv[i][c], kf[kk][c], acc);
        part[kk] = acc;
      }
      float s = reduce_scatter8(part, lane);
      const int pos = len - p.n_q + i;  // this query's position in its sequence
      const bool visible = my_key < c1 && my_key <= pos;
      s = visible ? s : -INFINITY;
      const float m_new = fmaxf(m[i], group_max(s));
      const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m[i] - m_new);
      const float pj = visible ? ex2_approx(s - m_new) : 0.f;
      l[i] = l[i] * alpha + group_sum(pj);
      m[i] = m_new;
#pragma unroll
      for (int c = 0; c < C; ++c) o[i][c] *= alpha;
#pragma unroll
      for (int kk = 0; kk < kGroup; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, pj, kk * 4);
#pragma unroll
        for (int c = 0; c < C; ++c) o[i][c] = fmaf(pk, vf[kk][c], o[i][c]);
      }
    }
  }

  // merge the warps of this CTA
#pragma unroll
  for (int i = 0; i < MAXQ; ++i) {
    if (lane == 0) {
      sm_m[warp][i] = m[i];
      sm_l[warp][i] = l[i];
    }
#pragma unroll
    for (int c = 0; c < C; ++c) sm_o[warp][i][lane * C + c] = o[i][c];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < p.n_q * D; idx += kDecThreads) {
    const int i = idx / D, col = idx % D;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, sm_m[w][i]);
    float ll = 0.f, oo = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float sc = (sm_m[w][i] == -INFINITY) ? 0.f : ex2_approx(sm_m[w][i] - mm);
      ll += sm_l[w][i] * sc;
      oo += sm_o[w][i][col] * sc;
    }
    const long long row = static_cast<long long>(bh) * p.n_q + i;
    if (p.splits == 1) {
      p.out[row * D + col] = to_bf16(ll > 0.f ? oo / ll : 0.f);
    } else {
      const long long slot = static_cast<long long>(split) * p.b * p.h * p.n_q + row;
      p.part_o[slot * D + col] = oo;
      if (col == 0) {
        p.part_ml[slot * 2 + 0] = mm;
        p.part_ml[slot * 2 + 1] = ll;
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(D) sdpa_decode_combine(const DecodeParams p) {
  griddep_wait();   // every split's partial results are complete
  const long long row = blockIdx.x;
  const int col = threadIdx.x;
  const long long rows = static_cast<long long>(p.b) * p.h * p.n_q;
  float mm = -INFINITY;
  for (int s = 0; s < p.splits; ++s) mm = fmaxf(mm, p.part_ml[(s * rows + row) * 2]);
  float ll = 0.f, oo = 0.f;
  for (int s = 0; s < p.splits; ++s) {
    const float ms = p.part_ml[(s * rows + row) * 2];
    const float sc = (ms == -INFINITY) ? 0.f : ex2_approx(ms - mm);
    ll += p.part_ml[(s * rows + row) * 2 + 1] * sc;
    oo += p.part_o[(s * rows + row) * D + col] * sc;
  }
  p.out[row * D + col] = to_bf16(ll > 0.f ? oo / ll : 0.f);
}

template <int D, int MAXQ>
cudaError_t launch_split(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(p.splits, p.b * p.h);
  sdpa_decode_split<D, MAXQ><<<grid, kDecThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t err;
  if (p.n_q == 1) err = launch_split<D, 1>(p, stream);
  else if (p.n_q <= 4) err = launch_split<D, 4>(p, stream);
  else err = launch_split<D, 8>(p, stream);
  if (err != cudaSuccess || p.splits == 1) return err;
  // programmatic dependency on the split kernel just launched
  return launch_kernel(sdpa_decode_combine<D>, dim3(static_cast<unsigned>(p.b * p.h * p.n_q)),
                       dim3(D), 0, stream, true, p);
}

}  // namespace

int decode_splits(int b, int h, int n_k) {
  const long long bh = static_cast<long long>(b) * h;
  if (bh <= 0 || n_k <= 0) return 1;
  long long s = (kDecodeTargetCtas + bh - 1) / bh;
  const long long by_len = (n_k + kDecodeMinKeysPerSplit - 1) / kDecodeMinKeysPerSplit;
  if (s > by_len) s = by_len;
  if (s > kDecodeMaxSplits) s = kDecodeMaxSplits;
  return s < 1 ? 1 : static_cast<int>(s);
}

cudaError_t launch_sdpa_decode(const DecodeParams& p, int head_dim, cudaStream_t stream) {
  if (p.b * p.h > 65535) return cudaErrorInvalidConfiguration;
  if (head_dim == 64) return launch_d<64>(p, stream);
  if (head_dim == 128) return launch_d<128>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
