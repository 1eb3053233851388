// bf16 GEMM on the GB300 tensor cores for the projections of multi-head
// attention ("Attention Is All You Need", section 3.2.2: Q W^Q, K W^K, V W^V
// and Concat(heads) W^O), Y = X W with X [m, k], W [k, n], Y [m, n] row-major.
//
// One CTA computes a 128 x BN tile of Y (BN = 256 or 128) with a single
// accumulator of BN fp32 columns in tensor memory; two CTAs share an SM, so
// one CTA's epilogue overlaps the other's products:
//   warp 0      TMA producer: 64-wide k-slices of X (K-major) and W (N
//               contiguous, i.e. MN-major for the MMA) into a ring of 2 or 3
//               stages (48 or 32 KB each).
//   warp 1      MMA issuer: tcgen05.mma M=128, N=BN, K=16, four per slice.
//   warps 2-5   epilogue: tensor memory -> registers -> bf16 -> swizzled
//               shared memory -> TMA store (clipped at the matrix edge).
// Up to three independent problems share one launch (blockIdx.z), which runs
// the Q, K and V projections together.  Measured on GB300, 128 x 256 tiles
// with two CTAs per SM are the fastest or within 1 us of it on every
// projection shape of the base and big models; 128-column tiles win only
// when 256-column ones would leave half the SMs idle (the base model's
// W^O, 4096 x 512 x 512).
#include <atomic>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int BM = kGemmBlockM;   // 128
constexpr int BK = 64;            // one 128-byte swizzle span of bf16
constexpr int kThreads = 192;
constexpr int kABytes = BM * BK * 2;           // 16 KB
constexpr int kBBoxBytes = BK * 64 * 2;        // 8 KB: 64 k-rows x 64 n
constexpr int kCBoxBytes = BM * 64 * 2;        // 16 KB staging box (128 rows x 64 cols)
constexpr int kMinBlocks = 2;                  // CTAs per SM

template <int BN>
struct GCfg {
  static constexpr int kStages = BN == 256 ? 2 : 3;
  static constexpr int kBBytes = BN * BK * 2;  // 32 or 16 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOff + (2 * kStages + 2) * 8 + 16 + 1024;
  static constexpr uint32_t kTmemCols = BN;
  static constexpr uint32_t kIdesc = idesc_bf16(BM, BN, false, true);
  static_assert(kSmemBytes * kMinBlocks <= 232448, "two CTAs per SM");
  static_assert((BN / 64) * kCBoxBytes <= kBarOff, "the epilogue stages Y over the ring");
};

template <int BN>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    gemm_bf16_tc(const __grid_constant__ GemmParams p) {
  using C = GCfg<BN>;
  constexpr int kStages = C::kStages;
  constexpr int kStageBytes = C::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t smem_base = smem_u32(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const AbortState ab{abort_flag, p.status};

  const int z = blockIdx.z;
  if (z >= p.num_problems) return;
  // Static parameter addresses only: the TMA reads the maps in place.
  const GemmProblem* prp = z == 0 ? &p.prob[0] : (z == 1 ? &p.prob[1] : &p.prob[2]);
  const CUtensorMap* tm_a = &prp->tm_a;
  const CUtensorMap* tm_b = &prp->tm_b;
  const CUtensorMap* tm_c = &prp->tm_c;
  const int pm = prp->m, pn = prp->n, pk = prp->k;
  const int m0 = blockIdx.y * BM;
  const int n0 = blockIdx.x * BN;
  if (m0 >= pm || n0 >= pn) return;   // uniform over the CTA
  const int num_kb = (pk + BK - 1) / BK;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every CTA holds its tensor memory now: the next kernel in the stream may
  // launch; this grid's inputs may come from the previous one, so wait for it.
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(tm_a);
      tma_prefetch_desc(tm_b);
      tma_prefetch_desc(tm_c);
      int issued = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kStages;
        const uint32_t use = static_cast<uint32_t>(kb / kStages);
        if (kb >= kStages && !mbar_wait(empty + s, (use - 1) & 1u, ab)) break;
        uint8_t* a_dst = smem + s * kStageBytes;
        uint8_t* b_dst = a_dst + kABytes;
        mbar_arrive_expect_tx(full + s, kStageBytes);
        tma_load_2d(tm_a, full + s, a_dst, kb * BK, m0);
#pragma unroll
        for (int nb = 0; nb < BN / 64; ++nb)
          tma_load_2d(tm_b, full + s, b_dst + nb * kBBoxBytes, n0 + nb * 64, kb * BK);
        issued = kb + 1;
      }
      for (int kb = max(0, issued - kStages); kb < issued; ++kb)
        mbar_wait_drain(full + kb % kStages, static_cast<uint32_t>(kb / kStages) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kStages;
        ok = mbar_wait(full + s, static_cast<uint32_t>(kb / kStages) & 1u, ab);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_base = smem_base + s * kStageBytes;
        const uint32_t b_base = a_base + kABytes;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t a = smem_desc_sw128(a_base + k * 32, 16, 1024);
          // W slice: 64 k-rows of 128 bytes per 64-column box; k step = 16 rows.
          const uint64_t b = smem_desc_sw128(b_base + k * 16 * 128, kBBoxBytes, 1024);
          mma_bf16_ss(tmem, a, b, C::kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(empty + s);
      }
      if (ok) mma_commit(acc_full);
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // epilogue warps 2..5: TMEM lane quarter = warp % 4
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true;
    if (num_kb > 0) {
      ok = mbar_wait_warp(acc_full, 0, ab);
      tc_fence_after();
    }
    // All stages are free once the accumulator is complete: stage the tile there.
    uint8_t* stage = smem;
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t o[32];
        if (num_kb > 0) {
          tmem_ld32(lane_base + c * 32, o);
          tmem_ld_wait();
          reg_fence(o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        uint8_t* box = stage + (c >> 1) * kCBoxBytes;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]), __uint_as_float(o[q4 * 8 + 1]));
          v.y = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]), __uint_as_float(o[q4 * 8 + 3]));
          v.z = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]), __uint_as_float(o[q4 * 8 + 5]));
          v.w = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]), __uint_as_float(o[q4 * 8 + 7]));
          const uint32_t chunk = static_cast<uint32_t>((c & 1) * 4 + q4);
          *reinterpret_cast<uint4*>(box + sw128_offset(static_cast<uint32_t>(row), chunk)) = v;
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (warp == 2 && lane == 0 && !*abort_flag) {
      for (int nb = 0; nb < BN / 64; ++nb) {
        if (n0 + nb * 64 >= pn) break;
        tma_store_2d(tm_c, stage + nb * kCBoxBytes, n0 + nb * 64, m0);
      }
      tma_store_commit();
      tma_store_wait_read();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN>
cudaError_t launch_bn(const GemmParams& p, int max_m, int max_n, cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(gemm_bf16_tc<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GCfg<BN>::kSmemBytes);
  if (err != cudaSuccess) return err;
  dim3 grid((max_n + BN - 1) / BN, (max_m + BM - 1) / BM, p.num_problems);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  return launch_kernel(gemm_bf16_tc<BN>, grid, dim3(kThreads), GCfg<BN>::kSmemBytes, stream,
                       p.pdl != 0, p);
}

// Tile width: 256 columns, or 128 when 256-column tiles would not reach
// half the SMs.  sdpa_set_kernel_choice can pin it to 256 or 128.
int gemm_tile_n(const GemmParams& p) {
  const int pin = gemm_bn_pin();
  if (pin == 256 || pin == 128) return pin;
  const int sms = device_sm_count();
  long long tiles = 0;
  for (int i = 0; i < p.num_problems; ++i)
    tiles += 1ll * ((p.prob[i].m + BM - 1) / BM) * ((p.prob[i].n + 255) / 256);
  return 2 * tiles >= sms ? 256 : 128;
}

}  // namespace

// SMs of the current device, read once per device.
int device_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 148;
  }
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      cudaGetLastError();
      return 148;
    }
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

cudaError_t launch_gemm_tc(const GemmParams& p, int max_m, int max_n, cudaStream_t stream) {
  if (max_m <= 0 || max_n <= 0 || p.num_problems <= 0) return cudaSuccess;
  const int bn = gemm_tile_n(p);
  if (bn == 256) return launch_bn<256>(p, max_m, max_n, stream);
  return launch_bn<128>(p, max_m, max_n, stream);
}

}  // namespace sdpa
