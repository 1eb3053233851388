// One autoregressive decoding step ("Attention Is All You Need", section 3.1:
// the decoder produces one symbol at a time): n_q <= 8 new queries per
// (batch, head) attend to a cached K/V of length len_b, query i seeing keys
// j <= len_b - n_q + i.  Eq. (1) with the causal rule of section 3.2.3, at
// every head shape of Table 3: d_k = d_v in {16, 32, 64, 128, 256, 512} and
// d_k in {16, 32} against d_v = 64 (rows (B)).
//
// The step reads every cached key and value once and does 2 (d_k + d_v) FLOP
// per key and query, so it is bound by HBM bandwidth, not by the tensor
// cores.  It runs on the CUDA cores and splits each sequence's cache across
// CTAs so the whole GPU streams it:
//   sdpa_decode_split   grid (splits, b*h), 4 warps.  Each warp walks its own
//                       tiles of TK keys of the CTA's key range, double
//                       buffered (single at d = 512, so that two CTAs fit an
//                       SM): one lane loads a tile's K and V rows with the
//                       TMA (rows swizzled at their width, as the attention
//                       kernels load them) while the warp works on the other.  Scores: each key of the tile belongs to
//                       LK lanes (one lane up to d_k = 64), which form its
//                       dot products with every query from their share of the
//                       columns; the queries sit in shared memory, pre-scaled
//                       to log2 units, and are read as broadcasts.  The
//                       swizzle puts the rows that neighbouring lanes read on
//                       different banks.  Softmax: one running max per query
//                       (a warp max per tile) and per-lane partial sums; the
//                       weights go to shared memory.  Values: each lane owns
//                       d_v / 32 contiguous output columns (for d_v = 16, two
//                       halves of the warp take alternate keys) and
//                       accumulates weight x value over the tile's keys with
//                       paired fp32 FMAs.  No lane exchanges anything per key.
//                       At the end the 4 warps merge through shared memory and
//                       the CTA writes the output (one split) or its partial
//                       (m, l, O) to the workspace.
//   sdpa_decode_combine merges the splits' partials: O = sum_s O_s 2^(m_s-M) /
//                       sum_s l_s 2^(m_s-M), M = max_s m_s.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = 32 * kDecWarps;

template <int DK, int DV, int MAXQ>
struct DCfg {
  static constexpr int LK = DK <= 64 ? 1 : (DK == 128 ? 2 : 4);   // lanes per key (scores)
  static constexpr int TK = 32 / LK;                                // keys per tile
  static constexpr int KCOLS = DK / LK;                             // key columns per lane
  static constexpr int KBOX = DK < 64 ? DK : 64;                    // columns per TMA box
  static constexpr int VBOX = DV < 64 ? DV : 64;
  static constexpr int KROW = KBOX * 2;                             // bytes per box row
  static constexpr int VROW = VBOX * 2;
  static constexpr int KBOXB = TK * KROW;                           // bytes per box
  static constexpr int VBOXB = TK * VROW;
  static constexpr int KBYTES = (DK / KBOX) * KBOXB;                // TK x DK x 2
  static constexpr int VBYTES = (DV / VBOX) * VBOXB;
  static constexpr int STAGE = KBYTES + VBYTES;
  // two stages per warp; one at d = 512 (16 KB a stage), so that two CTAs share an SM
  static constexpr int kStages = STAGE >= 16384 ? 1 : 2;
  // value columns: CV contiguous ones per lane; below 32 columns the warp
  // splits into KS slices of lanes that take alternate keys
  static constexpr int CV = DV >= 32 ? DV / 32 : 1;
  static constexpr int KS = DV >= 32 ? 1 : 32 / DV;
  static constexpr int QROW = KCOLS + 4;                            // floats per (query, part)
  // shared memory, from a 1024-byte aligned base
  static constexpr int kStageOff = 0;                               // [warp][stage]: K, V
  static constexpr int kQOff = kDecWarps * kStages * STAGE;
  static constexpr int kQBytes = MAXQ * LK * QROW * 4;
  static constexpr int kPOff = kQOff + kQBytes;                     // [warp][TK][MAXQ]
  static constexpr int kPBytes = kDecWarps * TK * MAXQ * 4;
  static constexpr int kBarOff = (kPOff + kPBytes + 7) / 8 * 8;
  static constexpr int kSmemBytes = kBarOff + kDecWarps * kStages * 8 + 16 + 1024;
  // the warps' merge reuses the stage buffers and the queries once every
  // tile is consumed
  static constexpr int kMergeBytes = kDecWarps * MAXQ * (DV + 2) * 4;
  static_assert(kMergeBytes <= kPOff, "merge buffer");
  static_assert(KBOXB % 1024 == 0 && VBOXB % 1024 == 0, "swizzle atoms");
  static_assert(DK % (8 * LK) == 0 && KCOLS % 8 == 0, "score chunks");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile of `box`-column
// boxes with rows of RowBytes, swizzled at that width: the column's box,
// then the row inside it.
template <int RowBytes, int BoxBytes>
__device__ __forceinline__ uint32_t tile_chunk(uint32_t row, uint32_t col) {
  constexpr uint32_t kColsPerBox = RowBytes / 2;
  const uint32_t box = col / kColsPerBox;
  const uint32_t chunk = (col % kColsPerBox) / 8;
  return box * BoxBytes + swizzle_offset<RowBytes>(row, chunk);
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
  return static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xffffu);
}

template <int DK, int DV, int MAXQ>
__global__ void __launch_bounds__(kDecThreads) sdpa_decode_split(const __grid_constant__ DecodeParams p) {
  using C = DCfg<DK, DV, MAXQ>;
  constexpr int TK = C::TK;
  constexpr int LK = C::LK;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  float* q_s = reinterpret_cast<float*>(smem + C::kQOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kDecWarps * C::kStages);
  const AbortState ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int bh = blockIdx.y;
  const int bi = bh / p.h;
  const int hi = bh % p.h;
  uint64_t* full = bars + warp * C::kStages;
  float* p_s = reinterpret_cast<float*>(smem + C::kPOff) + warp * TK * MAXQ;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecWarps * C::kStages; ++i) mbar_init(bars + i, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // the combine kernel may launch now; this grid's inputs may come from the
  // previous kernel in the stream, so wait for it before reading them
  griddep_launch_dependents();
  griddep_wait();
  int len = p.n_k;
  if (p.kv_lengths != nullptr) {
    len = p.kv_lengths[bi];
    len = len < 0 ? 0 : (len > p.n_k ? p.n_k : len);
  }
  // queries -> shared memory, fp32, scaled so that scores come out in log2
  // units; rows of each part of the columns padded by 4 floats
  for (int idx = threadIdx.x; idx < MAXQ * DK; idx += kDecThreads) {
    const int i = idx / DK, c = idx % DK;
    float x = 0.f;
    if (i < p.n_q) {
      const uint16_t u = p.q[(static_cast<long long>(bh) * p.n_q + i) * DK + c];
      x = __uint_as_float(static_cast<uint32_t>(u) << 16) * p.scale_log2;
    }
    q_s[(i * LK + c / C::KCOLS) * C::QROW + c % C::KCOLS] = x;
  }
  __syncthreads();

  const int c0 = split * p.keys_per_split;
  const int c1 = min(c0 + p.keys_per_split, len);
  const int n_tiles = c1 > c0 ? (c1 - c0 + TK - 1) / TK : 0;
  // this warp's tiles: t = warp, warp + kDecWarps, ...; local index u
  const int my_tiles = n_tiles > warp ? (n_tiles - warp + kDecWarps - 1) / kDecWarps : 0;
  auto tile_key = [&](int u) { return c0 + (warp + u * kDecWarps) * TK; };
  auto load_tile = [&](int u) {
    const int s = u % C::kStages;
    uint8_t* kst = smem + C::kStageOff + (warp * C::kStages + s) * C::STAGE;
    mbar_arrive_expect_tx(full + s, C::STAGE);
    const int j0 = tile_key(u);
#pragma unroll
    for (int c = 0; c < DK / C::KBOX; ++c)
      tma_load_4d(&p.tm_k, full + s, kst + c * C::KBOXB, c * C::KBOX, j0, hi, bi);
#pragma unroll
    for (int c = 0; c < DV / C::VBOX; ++c)
      tma_load_4d(&p.tm_v, full + s, kst + C::KBYTES + c * C::VBOXB, c * C::VBOX, j0, hi, bi);
  };
  if (lane == 0) {
    for (int u = 0; u < my_tiles && u < C::kStages; ++u) load_tile(u);
  }
  int issued = my_tiles < C::kStages ? my_tiles : C::kStages;

  // scores: key kj = lane / LK of the tile, columns [part * KCOLS, +KCOLS)
  const int kj = lane / LK;
  const int part = lane % LK;
  // values: columns [cg * CV, +CV), keys slice, slice + KS, ...
  const int cg = lane % (32 / C::KS);
  const int slice = lane / (32 / C::KS);
  float m[MAXQ], lsum[MAXQ], o[MAXQ][C::CV];
#pragma unroll
  for (int i = 0; i < MAXQ; ++i) {
    m[i] = -INFINITY;
    lsum[i] = 0.f;
#pragma unroll
    for (int c = 0; c < C::CV; ++c) o[i][c] = 0.f;
  }
  const int nq = p.n_q;
  bool ok = true;
  for (int u = 0; u < my_tiles; ++u) {
    const int s = u % C::kStages;
    if (!mbar_wait_warp(full + s, static_cast<uint32_t>(u / C::kStages) & 1u, ab)) {
      ok = false;
      break;
    }
    const uint8_t* kst = smem + C::kStageOff + (warp * C::kStages + s) * C::STAGE;
    const uint8_t* vst = kst + C::KBYTES;
    const int j0 = tile_key(u);

    // ---- scores of key kj against every query (log2 units)
    float2 acc[MAXQ];
#pragma unroll
    for (int i = 0; i < MAXQ; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < C::KCOLS; c += 8) {
      const int col = part * C::KCOLS + c;
      const uint4 kr = *reinterpret_cast<const uint4*>(
          kst + tile_chunk<C::KROW, C::KBOXB>(static_cast<uint32_t>(kj), static_cast<uint32_t>(col)));
      const float2 k0 = bf16x2_to_float2(kr.x), k1 = bf16x2_to_float2(kr.y);
      const float2 k2 = bf16x2_to_float2(kr.z), k3 = bf16x2_to_float2(kr.w);
#pragma unroll
      for (int i = 0; i < MAXQ; ++i) {
        const float4* qp = reinterpret_cast<const float4*>(q_s + (i * LK + part) * C::QROW + c);
        const float4 qa = qp[0], qb = qp[1];
        acc[i] = __ffma2_rn(k0, make_float2(qa.x, qa.y), acc[i]);
        acc[i] = __ffma2_rn(k1, make_float2(qa.z, qa.w), acc[i]);
        acc[i] = __ffma2_rn(k2, make_float2(qb.x, qb.y), acc[i]);
        acc[i] = __ffma2_rn(k3, make_float2(qb.z, qb.w), acc[i]);
      }
    }
    const int key = j0 + kj;
    float alpha[MAXQ];
#pragma unroll
    for (int i = 0; i < MAXQ; ++i) {
      float sc = acc[i].x + acc[i].y;
#pragma unroll
      for (int x = 1; x < LK; x <<= 1) sc += __shfl_xor_sync(0xffffffffu, sc, x);
      // query i sits at position len - n_q + i and sees keys up to it
      const bool visible = i < nq && key < c1 && key <= len - nq + i;
      sc = visible ? sc : -INFINITY;
      float tmax = sc;
#pragma unroll
      for (int x = 1; x < 32; x <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, x));
      const float m_new = fmaxf(m[i], tmax);
      alpha[i] = (m_new == -INFINITY) ? 1.f : ex2_approx(m[i] - m_new);
      const float pw = visible ? ex2_approx(sc - m_new) : 0.f;
      m[i] = m_new;
      lsum[i] = lsum[i] * alpha[i] + (part == 0 ? pw : 0.f);
      if (part == 0) p_s[kj * MAXQ + i] = pw;
    }
    __syncwarp();

    // ---- O += P V over the tile's keys, this lane's columns
#pragma unroll
    for (int i = 0; i < MAXQ; ++i)
#pragma unroll
      for (int c = 0; c < C::CV; ++c) o[i][c] *= alpha[i];
#pragma unroll 4
    for (int j = slice; j < TK; j += C::KS) {
      float pj[MAXQ];
      if constexpr (MAXQ % 4 == 0) {
#pragma unroll
        for (int i = 0; i < MAXQ; i += 4) {
          const float4 t = *reinterpret_cast<const float4*>(p_s + j * MAXQ + i);
          pj[i] = t.x; pj[i + 1] = t.y; pj[i + 2] = t.z; pj[i + 3] = t.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < MAXQ; ++i) pj[i] = p_s[j * MAXQ + i];
      }
      const uint8_t* vrow = vst + tile_chunk<C::VROW, C::VBOXB>(
                                      static_cast<uint32_t>(j), static_cast<uint32_t>(cg * C::CV));
      const uint32_t byte_in_chunk = (cg * C::CV * 2) % 16;
      if constexpr (C::CV >= 8) {
        // whole 16-byte chunks: CV / 8 of them, contiguous in the logical row
#pragma unroll
        for (int h = 0; h < C::CV / 8; ++h) {
          const uint8_t* src = vst + tile_chunk<C::VROW, C::VBOXB>(
                                         static_cast<uint32_t>(j),
                                         static_cast<uint32_t>(cg * C::CV + h * 8));
          const uint4 vr = *reinterpret_cast<const uint4*>(src);
          const float2 v0 = bf16x2_to_float2(vr.x), v1 = bf16x2_to_float2(vr.y);
          const float2 v2 = bf16x2_to_float2(vr.z), v3 = bf16x2_to_float2(vr.w);
#pragma unroll
          for (int i = 0; i < MAXQ; ++i) {
            const float2 pp = make_float2(pj[i], pj[i]);
            float2* oo = reinterpret_cast<float2*>(&o[i][h * 8]);
            oo[0] = __ffma2_rn(pp, v0, oo[0]);
            oo[1] = __ffma2_rn(pp, v1, oo[1]);
            oo[2] = __ffma2_rn(pp, v2, oo[2]);
            oo[3] = __ffma2_rn(pp, v3, oo[3]);
          }
        }
      } else if constexpr (C::CV == 4) {
        const uint2 vr = *reinterpret_cast<const uint2*>(vrow + byte_in_chunk);
        const float2 v0 = bf16x2_to_float2(vr.x), v1 = bf16x2_to_float2(vr.y);
#pragma unroll
        for (int i = 0; i < MAXQ; ++i) {
          const float2 pp = make_float2(pj[i], pj[i]);
          float2* oo = reinterpret_cast<float2*>(&o[i][0]);
          oo[0] = __ffma2_rn(pp, v0, oo[0]);
          oo[1] = __ffma2_rn(pp, v1, oo[1]);
        }
      } else if constexpr (C::CV == 2) {
        const float2 v0 = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vrow + byte_in_chunk));
#pragma unroll
        for (int i = 0; i < MAXQ; ++i) {
          float2* oo = reinterpret_cast<float2*>(&o[i][0]);
          oo[0] = __ffma2_rn(make_float2(pj[i], pj[i]), v0, oo[0]);
        }
      } else {
        const uint16_t vb = *reinterpret_cast<const uint16_t*>(vrow + byte_in_chunk);
        const float v0 = __uint_as_float(static_cast<uint32_t>(vb) << 16);
#pragma unroll
        for (int i = 0; i < MAXQ; ++i) o[i][0] = fmaf(pj[i], v0, o[i][0]);
      }
    }
    // every lane is done with this stage and with the weights: refill it
    __syncwarp();
    if (lane == 0 && issued < my_tiles) {
      fence_proxy_async_smem();
      load_tile(issued);
    }
    ++issued;
  }
  // a timed-out wait leaves at most the stages' last loads in flight: let
  // them land before the buffers are reused or the CTA exits
  if (!ok && lane == 0) {
    const int last = (issued < my_tiles ? issued : my_tiles);
    for (int u = last - C::kStages < 0 ? 0 : last - C::kStages; u < last; ++u)
      mbar_wait_drain(full + u % C::kStages, static_cast<uint32_t>(u / C::kStages) & 1u);
  }

  // ---- per-warp totals: the row sums over lanes (one lane per key counted),
  // and for d_v < 32 the key slices' partial outputs
#pragma unroll
  for (int i = 0; i < MAXQ; ++i) {
#pragma unroll
    for (int x = 1; x < 32; x <<= 1) lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], x);
    if constexpr (C::KS > 1) {
#pragma unroll
      for (int x = 32 / C::KS; x < 32; x <<= 1)
#pragma unroll
        for (int c = 0; c < C::CV; ++c) o[i][c] += __shfl_xor_sync(0xffffffffu, o[i][c], x);
    }
  }
  __syncthreads();   // every warp is done with its stages: reuse them for the merge
  float* mg_o = reinterpret_cast<float*>(smem + C::kStageOff);      // [warp][MAXQ][DV]
  float* mg_ml = mg_o + kDecWarps * MAXQ * DV;                      // [warp][MAXQ][2]
#pragma unroll
  for (int i = 0; i < MAXQ; ++i) {
    if (lane == 0) {
      mg_ml[(warp * MAXQ + i) * 2] = ok ? m[i] : -INFINITY;
      mg_ml[(warp * MAXQ + i) * 2 + 1] = ok ? lsum[i] : 0.f;
    }
    if (slice == 0) {
#pragma unroll
      for (int c = 0; c < C::CV; ++c) mg_o[(warp * MAXQ + i) * DV + cg * C::CV + c] = o[i][c];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nq * DV; idx += kDecThreads) {
    const int i = idx / DV, col = idx % DV;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, mg_ml[(w * MAXQ + i) * 2]);
    float ll = 0.f, oo = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float mw = mg_ml[(w * MAXQ + i) * 2];
      const float sc = (mw == -INFINITY) ? 0.f : ex2_approx(mw - mm);
      ll += mg_ml[(w * MAXQ + i) * 2 + 1] * sc;
      oo += mg_o[(w * MAXQ + i) * DV + col] * sc;
    }
    const long long row = static_cast<long long>(bh) * p.n_q + i;
    if (p.splits == 1) {
      p.out[row * DV + col] = to_bf16(ll > 0.f ? oo / ll : 0.f);
    } else {
      const long long slot = static_cast<long long>(split) * p.b * p.h * p.n_q + row;
      p.part_o[slot * DV + col] = oo;
      if (col == 0) {
        p.part_ml[slot * 2 + 0] = mm;
        p.part_ml[slot * 2 + 1] = ll;
      }
    }
  }
}

template <int DV>
__global__ void __launch_bounds__(DV) sdpa_decode_combine(const DecodeParams p) {
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
    oo += p.part_o[(s * rows + row) * DV + col] * sc;
  }
  p.out[row * DV + col] = to_bf16(ll > 0.f ? oo / ll : 0.f);
}

template <int DK, int DV, int MAXQ>
cudaError_t launch_split(const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = DCfg<DK, DV, MAXQ>::kSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(sdpa_decode_split<DK, DV, MAXQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  // a programmatic dependency on the previous kernel: the split kernel reads
  // its inputs only after griddep_wait()
  return launch_kernel(sdpa_decode_split<DK, DV, MAXQ>, dim3(p.splits, p.b * p.h),
                       dim3(kDecThreads), smem, stream, true, p);
}

template <int DK, int DV>
cudaError_t launch_shape(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t err;
  if (p.n_q == 1) err = launch_split<DK, DV, 1>(p, stream);
  else if (p.n_q <= 4) err = launch_split<DK, DV, 4>(p, stream);
  else err = launch_split<DK, DV, 8>(p, stream);
  if (err != cudaSuccess || p.splits == 1) return err;
  // programmatic dependency on the split kernel just launched
  return launch_kernel(sdpa_decode_combine<DV>, dim3(static_cast<unsigned>(p.b * p.h * p.n_q)),
                       dim3(DV), 0, stream, true, p);
}

template <int DK, int DV>
int resident_ctas() {
  // CTAs of the largest-query variant that share an SM (shared memory bound)
  constexpr int smem = DCfg<DK, DV, 8>::kSmemBytes + 1024;
  const int by_smem = 232448 / smem;
  return by_smem < 1 ? 1 : (by_smem > kDecodeMaxResident ? kDecodeMaxResident : by_smem);
}

}  // namespace

bool decode_supports(int d_k, int d_v) {
  if (d_k == d_v)
    return d_k == 16 || d_k == 32 || d_k == 64 || d_k == 128 || d_k == 256 || d_k == 512;
  return d_v == 64 && (d_k == 16 || d_k == 32);
}

int decode_keys_per_tile(int d_k) { return d_k <= 64 ? 32 : (d_k == 128 ? 16 : 8); }

int decode_resident_ctas(int d_k, int d_v) {
  if (d_k != d_v) return d_k == 16 ? resident_ctas<16, 64>() : resident_ctas<32, 64>();
  switch (d_k) {
    case 16: return resident_ctas<16, 16>();
    case 32: return resident_ctas<32, 32>();
    case 64: return resident_ctas<64, 64>();
    case 128: return resident_ctas<128, 128>();
    case 256: return resident_ctas<256, 256>();
    default: return resident_ctas<512, 512>();
  }
}

int decode_splits(int b, int h, int n_k, int target_ctas) {
  const long long bh = static_cast<long long>(b) * h;
  if (bh <= 0 || n_k <= 0) return 1;
  long long s = (target_ctas + bh - 1) / bh;
  const long long by_len = (n_k + kDecodeMinKeysPerSplit - 1) / kDecodeMinKeysPerSplit;
  if (s > by_len) s = by_len;
  if (s > kDecodeMaxSplits) s = kDecodeMaxSplits;
  return s < 1 ? 1 : static_cast<int>(s);
}

cudaError_t launch_sdpa_decode(const DecodeParams& p, int d_k, int d_v, cudaStream_t stream) {
  if (p.b * p.h > 65535) return cudaErrorInvalidConfiguration;
  if (d_k != d_v) {
    if (d_v != 64) return cudaErrorInvalidValue;
    if (d_k == 16) return launch_shape<16, 64>(p, stream);
    if (d_k == 32) return launch_shape<32, 64>(p, stream);
    return cudaErrorInvalidValue;
  }
  switch (d_k) {
    case 16: return launch_shape<16, 16>(p, stream);
    case 32: return launch_shape<32, 32>(p, stream);
    case 64: return launch_shape<64, 64>(p, stream);
    case 128: return launch_shape<128, 128>(p, stream);
    case 256: return launch_shape<256, 256>(p, stream);
    case 512: return launch_shape<512, 512>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sdpa
