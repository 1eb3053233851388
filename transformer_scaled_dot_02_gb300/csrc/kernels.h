// Host-side launch interfaces of the CUDA kernels (internal to libsdpa).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace sdpa {

// Error bits of the device status word (read back by sdpa_device_check).
constexpr unsigned kStatusTimeout = 1u;

// Fused bf16 attention on the tensor cores.  The four tensor maps view
// Q, K, V and O as 4-D (d, n, h, b) arrays with 64 x 128 boxes, 128-byte
// swizzle; any strides for n, h, b (BHSD inputs, or BSHD inside the
// multi-head path).
struct SdpaTcParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  const int32_t* kv_lengths;  // device [b] or null
  unsigned* status;           // device error word
  int b, h, n_q, n_k;
  int mask_kind;
  int num_q_blocks;           // ceil(n_q / 256)
  float scale_log2;           // scale * log2(e)
  // Restricted attention: query i sees keys [i - win_left, i + win_right]
  // (kWindowUnbounded for plain attention).
  int win_left, win_right;
  float* lse;                 // optional [b, h, n_q] natural log-sum-exp per row
  int pdl = 0;                // launched with a programmatic dependency on the previous kernel
  // One-tile kernel: CTAs take (head, d_v slice) units in groups of this
  // many, the longest query tiles of a group first (>= 1).
  int head_group = 8;
};
constexpr int kWindowUnbounded = 1 << 30;

// Launches `kernel` on `stream`; with `pdl` it may start (and run its set-up)
// while the previous kernel in the stream finishes: the kernels call
// griddep_launch_dependents() once their tensor memory is allocated and
// griddep_wait() before touching global memory the previous kernel writes.
template <typename Params>
inline cudaError_t launch_kernel(void (*kernel)(Params), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool pdl, const Params& p) {
  if (!pdl) {
    kernel<<<grid, block, smem, stream>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}
// Two query tiles per CTA; (d_k, d_v) in {(16,16), (32,32), (64,64), (128,128), (16,64), (32,64)}.
cudaError_t launch_sdpa_tc(const SdpaTcParams& p, int d_k, int d_v, cudaStream_t stream);
// One 128-row query tile per CTA (d = 16 .. 512) with key tiles of key_tile
// rows (32 for d = 16, 32; 32 or 64 for d = 64; 64 from d = 128); the K/V
// maps' boxes must have key_tile rows; num_q_blocks = ceil(n_q / 128).
bool one_tile_supports(int head_dim, int key_tile);
cudaError_t launch_sdpa_one_tile(const SdpaTcParams& p, int head_dim, int key_tile,
                                 cudaStream_t stream);

// SMs of the current device (read once per device and cached).
int device_sm_count();

// Column tile of the projection GEMM pinned by sdpa_set_kernel_choice (0: by shape).
int gemm_bn_pin();

// One decoding step over a K/V cache on the CUDA cores, split across CTAs.
struct DecodeParams {
  CUtensorMap tm_k, tm_v;     // 4-D (d, n, h, b) bf16 maps of the caches, boxes of
                              // min(d, 64) columns x decode_keys_per_tile(d_k) rows
  const uint16_t* q;          // bf16 [b,h,n_q,d_k]
  uint16_t* out;              // bf16 [b,h,n_q,d_v]
  float* part_o;              // [splits][b*h*n_q][d_v]  (splits > 1)
  float* part_ml;             // [splits][b*h*n_q][2]  (splits > 1)
  const int32_t* kv_lengths;  // device [b] or null
  unsigned* status;           // device error word
  int b, h, n_q, n_k;
  int splits, keys_per_split;
  float scale_log2;
};
constexpr int kDecodeMaxQueries = 8;
constexpr int kDecodeMinKeysPerSplit = 256;
constexpr int kDecodeMaxSplits = 256;
constexpr int kDecodeWaves = 4;             // split CTAs: about this many waves of resident CTAs
constexpr int kDecodeMaxResident = 4;       // resident split CTAs per SM, at most
// (d_k, d_v) pairs the decode kernels are built for: every Table 3 head shape.
bool decode_supports(int d_k, int d_v);
// Keys per tile (TMA box rows) of the decode kernel for a key size.
int decode_keys_per_tile(int d_k);
// Split CTAs of one shape that share an SM.
int decode_resident_ctas(int d_k, int d_v);
// Splits of each sequence's cache for about target_ctas CTAs in all (each
// split at least kDecodeMinKeysPerSplit keys, at most kDecodeMaxSplits).
int decode_splits(int b, int h, int n_k, int target_ctas);
cudaError_t launch_sdpa_decode(const DecodeParams& p, int d_k, int d_v, cudaStream_t stream);

// Gradients of attention (bf16 BHSD tensors, fp32 accumulation).
struct SdpaBwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;   // 4-D (d, n, h, b) bf16 maps; d = d_k for Q, K
  CUtensorMap tm_dq;          // 3-D (d_k, n_q, b*h) fp32 map of dq_acc, 32-column boxes
  const float* neg_lse2;      // [b*h][n_q_pad] -lse_i log2(e) (-inf past n_q)
  const float* neg_dvec;      // [b*h][n_q_pad] -D_i = -dO_i . O_i
  float* dq_acc;              // [b*h][n_q][d_k] fp32 accumulator (zeroed by the prep kernel)
  uint16_t *dk, *dv;          // [b*h][n_k][d_k], [b*h][n_k][d_v] bf16 outputs
  const int32_t* kv_lengths;
  unsigned* status;
  int b, h, n_q, n_k, n_q_pad, mask_kind, num_kv_tiles;
  float scale_log2, scale;
  int win_left, win_right;
};
struct SdpaBwdPrepParams {
  const uint16_t *out, *dout;  // forward output and its gradient, [b*h][n_q][d_v]
  const float* lse;            // [b*h][n_q] natural log-sum-exp
  float *neg_lse2, *neg_dvec, *dq_acc;
  uint16_t* dq;                // [b*h][n_q][d_k] bf16 output
  int b, h, n_q, n_q_pad;
  float scale;
};
cudaError_t launch_sdpa_bwd(const SdpaBwdParams& bp, const SdpaBwdPrepParams& pp, int d_k, int d_v,
                            cudaStream_t stream);
// Key rows per CTA (the K / V boxes' rows, and n_k's tile size) and query rows
// per step (the Q / dO boxes' and the dQ reduce boxes' rows) of the backward
// for a head size: 128 and 64, or 64 and 32 for 512-wide heads.
int bwd_key_tile(int d_k);
int bwd_query_step(int d_k);
// The main kernel for 512-wide heads (after the prep kernel when `after_prep`).
cudaError_t launch_sdpa_bwd_w512(const SdpaBwdParams& bp, bool after_prep, cudaStream_t stream);
#ifdef __CUDACC__
// The steps [lo, hi) of Step queries that hold a query able to see one of the
// Keys keys from key0 (below kv_len), under the causal mask and the window.
template <int Keys, int Step>
__device__ __forceinline__ int2 bwd_query_steps(const SdpaBwdParams& p, int key0, int kv_len) {
  const int key_hi = min(key0 + Keys, kv_len) - 1;
  if (key_hi < key0) return make_int2(0, 0);
  long long q_lo = static_cast<long long>(key0) - p.win_right;
  if (p.mask_kind & 1) q_lo = q_lo > key0 ? q_lo : key0;
  if (q_lo < 0) q_lo = 0;
  long long q_hi = static_cast<long long>(key_hi) + p.win_left + 1;
  if (q_hi > p.n_q) q_hi = p.n_q;
  if (q_hi <= q_lo) return make_int2(0, 0);
  return make_int2(static_cast<int>(q_lo / Step), static_cast<int>((q_hi + Step - 1) / Step));
}
#endif

// Exact fp32 attention on the CUDA cores, BHSD contiguous.
struct SdpaF32Params {
  const float *q, *k, *v;
  float* out;
  const int32_t* kv_lengths;
  int b, h, n_q, n_k, d_k, d_v;
  int mask_kind;
  float scale;
};
cudaError_t launch_sdpa_f32(const SdpaF32Params& p, cudaStream_t stream);

// bf16 GEMM on the tensor cores, up to three independent problems per launch
// (blockIdx.z): Y[m, n] = X[m, k] * W[k, n], all row-major.
struct GemmProblem {
  CUtensorMap tm_a;  // X: 2-D (k, m), box 64 x 128, 128-byte swizzle
  CUtensorMap tm_b;  // W: 2-D (n, k), box 64 x 64, 128-byte swizzle
  CUtensorMap tm_c;  // Y: 2-D (n, m), box 64 x 128, 128-byte swizzle
  int m, n, k;
};
struct GemmParams {
  GemmProblem prob[3];
  int num_problems;
  unsigned* status;
  int pdl = 0;                // launched with a programmatic dependency on the previous kernel
};
constexpr int kGemmBlockM = 128;
cudaError_t launch_gemm_tc(const GemmParams& p, int max_m, int max_n, cudaStream_t stream);

}  // namespace sdpa
