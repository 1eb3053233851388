// Gradients of scaled dot-product attention for 512-wide heads ("Attention
// Is All You Need", section 5 through Eq. (1) of section 3.2.1; Table 3,
// row (A): one head of 512).  The same products as the narrower backward:
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,
// with P recomputed from the forward's log-sum-exp.
//
// At d = 512 a 128-key tile's K and V alone would take 256 KB of shared
// memory, so a CTA here owns 64 keys (K and V resident, 128 KB) and one half
// (256 columns) of d for its outputs; the two CTAs of a key tile both compute
// the scores.  The score products run with M = 64, which puts key r in
// tensor-memory lane (r mod 16) + 32 (r / 16): 16 lanes of each warp's quarter
// (measured on GB300).  They read half the A bytes of an M = 128 product,
// and shared-memory operand reads are what bound these small products.
// dV and dK accumulate transposed, d in the tensor-memory lanes, so the half's
// 256 columns of both take 256 tensor-memory columns:
//   S^T = K Q^T,  dP^T = V dO^T        (M = 64 keys, N = 32 queries, K = 512)
//   dV^T += dO^T P,  dK^T += Q^T dS    (M = 128 of d, N = 64 keys, K = 32 queries)
//   dQ^T = K^T dS^T                    (M = 128 of d, N = 32 queries, K = 64 keys)
// P and dS go through shared memory as [key][query] rows.  Queries come in
// steps of 32, each step's Q and dO in four parts (the half's own columns and
// the others, of each), so the next step's loads run while this step's
// products do: a part is refilled as soon as the last product reading it is
// done.  dQ leaves each step as tensor reduce-adds into the fp32 accumulator
// that the prep kernel zeroed; the convert kernel scales and rounds it.
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {
namespace {
namespace w512 {

constexpr int kD = 512;
constexpr int kKeys = 64;                      // keys per CTA
constexpr int kBN = 32;                        // queries per step
constexpr int kBoxCols = 64;                   // 128-byte swizzled rows
constexpr int kBoxes = kD / kBoxCols;          // 8 column boxes
constexpr int kHalfBoxes = kBoxes / 2;         // boxes of the CTA's half of d
constexpr int kKVBox = kKeys * 128;            // 64 keys x 64 columns: 8 KB
constexpr int kQBox = kBN * 128;               // 32 queries x 64 columns: 4 KB
constexpr int kPart = kHalfBoxes * kQBox;      // four boxes of Q or dO: 16 KB
constexpr int kKOff = 0;
constexpr int kVOff = kKOff + kBoxes * kKVBox;             // 64 KB
constexpr int kQnOff = kVOff + kBoxes * kKVBox;            // 128 KB: Q, the other half's boxes
constexpr int kQhOff = kQnOff + kPart;                     // Q, this half's boxes
constexpr int kDonOff = kQhOff + kPart;                    // dO, the other half's boxes
constexpr int kDohOff = kDonOff + kPart;                   // dO, this half's boxes
constexpr int kPOff = kDohOff + kPart;                     // 192 KB: P^T [64 keys][128 B]
constexpr int kDsOff = kPOff + kKeys * 128;                // dS^T, same layout
constexpr int kStagingWarp = kBN * 32 * 4;                 // [32 rows][32 columns] fp32
constexpr int kStagingOff = kDsOff + kKeys * 128;          // 208 KB: one per epilogue warp
constexpr int kVecBytes = 2 * kBN * 4;                     // -lse2 and -D of one step
// Three steps' vectors: step it + 2's are loaded once the scores of step
// it + 1 over the other half have read their Q part, which can be before the
// softmax of step it has read step it's; step it + 3's only after it has.
constexpr int kVecSlots = 3;
constexpr int kVecOff = kStagingOff + 4 * kStagingWarp;    // 224 KB
constexpr int kBarOff = kVecOff + kVecSlots * kVecBytes;
// kv_full, full[4], empty[4], vec_full[3], s_full, p_full, dq_full[2],
// dq_empty[2], acc_full, drain
constexpr int kNumBars = 1 + 4 + 4 + kVecSlots + 1 + 1 + 2 + 2 + 1 + 1;
constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kQnOff % 1024 == 0 && kPOff % 1024 == 0 && kStagingOff % 1024 == 0, "align");

// Warps: 0..7 compute (lanes 0..15 of quarter w % 4 hold keys 16 (w % 4) ..
// +16; query half w / 4); 8 TMA producer; 9 MMA issuer; 10..13 dQ^T and, at
// the end, dV and dK out of tensor memory (lane quarter w % 4).
constexpr int kThreads = 448;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kEpilogueWarp0 = 10;
constexpr int kCompute = 256;
constexpr int kEpilogue = 128;
constexpr int kHeadGroup = 2;     // heads whose key tiles run together (Q, dO, dQ stay in L2)

// Tensor-memory columns.  Two score buffers (step parity): the next step's
// scores over the other half's boxes run while the softmax works on this
// step's.
constexpr uint32_t kColS = 0;        // S^T at kColS + 64 b, 32 columns (M = 64 layout)
constexpr uint32_t kColDP = 32;      // dP^T at kColDP + 64 b
constexpr uint32_t kColDV = 128;     // dV^T: two 128-lane blocks of d x 64 keys
constexpr uint32_t kColDK = 256;     // dK^T
constexpr uint32_t kColDQ = 384;     // dQ^T: two buffers of (two blocks x 32 queries)

constexpr uint32_t kIdescS = idesc_bf16(kKeys, kBN, false, false);   // S^T, dP^T (M = 64)
constexpr uint32_t kIdescG = idesc_bf16(128, kKeys, true, false);    // dV^T, dK^T
constexpr uint32_t kIdescQ = idesc_bf16(128, kBN, true, true);       // dQ^T
// every operand: 128-byte swizzle, 8-row groups 1024 bytes apart
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);

__device__ __forceinline__ uint32_t desc_lo(uint32_t addr, uint32_t lbo) {
  return (addr >> 4) | ((lbo >> 4) << 16);
}

// Column box of part box j: this half's boxes (own) or the other half's.
__device__ __forceinline__ int part_box(int half, bool own, int j) {
  return (own ? half : 1 - half) * kHalfBoxes + j;
}

__global__ void __launch_bounds__(kThreads, 1) sdpa_bwd_tc_w512(const __grid_constant__ SdpaBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t smem_base = smem_u32(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* kv_full = bar;
  uint64_t* full = bar + 1;        // Q other, Q own, dO other, dO own
  uint64_t* empty = full + 4;
  uint64_t* vec_full = empty + 4;
  uint64_t* s_full = vec_full + kVecSlots;
  uint64_t* p_full = s_full + 1;
  uint64_t* dq_full = p_full + 1;
  uint64_t* dq_empty = dq_full + 2;
  uint64_t* acc_full = dq_empty + 2;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const AbortState ab{abort_flag, p.status};
  // part index (and order in shared memory): 0 = Q other, 1 = Q own,
  // 2 = dO other, 3 = dO own
  constexpr int kQo = 0, kQh = 1, kDo = 2, kDh = 3;
  static_assert(kQhOff == kQnOff + kPart && kDonOff == kQnOff + 2 * kPart &&
                    kDohOff == kQnOff + 3 * kPart, "parts in index order");
  auto part_off = [](int s) { return kQnOff + s * kPart; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh_count = p.b * p.h;
  // half of d, then heads in groups of kHeadGroup, each group's key tiles in
  // ascending order (the longest causal walks first)
  const int half = static_cast<int>(blockIdx.x) & 1;
  const int idx = static_cast<int>(blockIdx.x) >> 1;
  const int group_ctas = kHeadGroup * p.num_kv_tiles;
  const int full_groups = bh_count / kHeadGroup;
  int g = idx / group_ctas;
  int rr = idx % group_ctas;
  int heads_in_group = kHeadGroup;
  if (g >= full_groups) {
    g = full_groups;
    rr = idx - full_groups * group_ctas;
    heads_in_group = bh_count - full_groups * kHeadGroup;
  }
  const int jt = rr / heads_in_group;
  const int bh = g * kHeadGroup + rr % heads_in_group;
  const int bi = bh / p.h;
  const int hi = bh % p.h;
  const bool causal = (p.mask_kind & 1) != 0;
  // the caller's lengths: the prep kernel never writes them
  int kv_len = p.n_k;
  if ((p.mask_kind & 2) && p.kv_lengths != nullptr) {
    kv_len = p.kv_lengths[bi];
    kv_len = kv_len < 0 ? 0 : (kv_len > p.n_k ? p.n_k : kv_len);
  }
  const int key0 = jt * kKeys;
  const int2 qr = bwd_query_steps<kKeys, kBN>(p, key0, kv_len);
  const int i_lo = qr.x, n_it = qr.y - qr.x;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int v = 0; v < kVecSlots; ++v) mbar_init(vec_full + v, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(dq_full + b, 1);
      mbar_init(dq_empty + b, kEpilogue);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, kCompute);
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();

  if (warp == kProducerWarp) {
    if (lane == 0 && n_it > 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      mbar_arrive_expect_tx(kv_full, 2 * kBoxes * kKVBox);
      for (int c = 0; c < kBoxes; ++c)
        tma_load_4d(&p.tm_k, kv_full, smem + kKOff + c * kKVBox, c * kBoxCols, key0, hi, bi);
      for (int c = 0; c < kBoxes; ++c)
        tma_load_4d(&p.tm_v, kv_full, smem + kVOff + c * kKVBox, c * kBoxCols, key0, hi, bi);
      int issued[4] = {0, 0, 0, 0};
      int vec_issued = 0;
      bool go = true;
      for (int it = 0; go && it < n_it; ++it) {
        const int q0 = (i_lo + it) * kBN;
        // parts in the order their previous contents are released:
        // Q other, dO other, Q own, dO own
#pragma unroll
        for (int o = 0; o < 4; ++o) {
          const int s = ((o & 1) << 1) | (o >> 1);
          if (it > 0 && !mbar_wait(empty + s, static_cast<uint32_t>(it - 1) & 1u, ab)) {
            go = false;
            break;
          }
          const CUtensorMap* map = (s == kQo || s == kQh) ? &p.tm_q : &p.tm_do;
          const bool own = s == kQh || s == kDh;
          mbar_arrive_expect_tx(full + s, kPart);
          for (int j = 0; j < kHalfBoxes; ++j)
            tma_load_4d(map, full + s, smem + part_off(s) + j * kQBox,
                        part_box(half, own, j) * kBoxCols, q0, hi, bi);
          issued[s] = it + 1;
          if (s == kQo) {
            // this step's -lse2 and -D into slot it % 3; the slot's last
            // reader (the softmax of step it - 3) finished before the scores
            // of step it - 1 over the other half were issued, and those
            // released this Q part
            uint64_t* vb = vec_full + it % kVecSlots;
            uint8_t* vec = smem + kVecOff + (it % kVecSlots) * kVecBytes;
            const long long vrow = static_cast<long long>(bh) * p.n_q_pad + q0;
            mbar_arrive_expect_tx(vb, kVecBytes);
            tma_load_1d(vec, p.neg_lse2 + vrow, kBN * 4, vb);
            tma_load_1d(vec + kBN * 4, p.neg_dvec + vrow, kBN * 4, vb);
            vec_issued = it + 1;
          }
        }
      }
      // let the copies still in flight land before the CTA can exit
      mbar_wait_drain(kv_full, 0);
      for (int s = 0; s < 4; ++s)
        if (issued[s] > 0) mbar_wait_drain(full + s, static_cast<uint32_t>(issued[s] - 1) & 1u);
      for (int it = vec_issued > kVecSlots ? vec_issued - kVecSlots : 0; it < vec_issued; ++it)
        mbar_wait_drain(vec_full + it % kVecSlots, static_cast<uint32_t>(it / kVecSlots) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // The whole warp runs this loop in step; one elected lane issues.
    if (n_it > 0) {
      // S^T (dp false) or dP^T (dp true) of step `it` over the four boxes of
      // one part, into the step's score buffer; `first` starts the accumulation
      auto scores = [&](int it, bool dp, bool own, bool first) {
        const uint32_t a_base = smem_base + (dp ? kVOff : kKOff);
        const uint32_t b_base = smem_base + part_off(dp ? (own ? kDh : kDo) : (own ? kQh : kQo));
        const uint32_t d = tmem + (dp ? kColDP : kColS) + static_cast<uint32_t>((it & 1) * 64);
#pragma unroll
        for (int j = 0; j < kHalfBoxes; ++j) {
          const uint32_t a0 = desc_lo(a_base + part_box(half, own, j) * kKVBox, 16);
          const uint32_t b0 = desc_lo(b_base + j * kQBox, 16);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ss_warp(d, a0 + static_cast<uint32_t>(k * 2), kDescHi,
                             b0 + static_cast<uint32_t>(k * 2), kDescHi, kIdescS,
                             (first && j == 0 && k == 0) ? 0u : 1u);
        }
      };
      // The scores of step it over the other half's boxes (their loads
      // started earliest), then over this half's, which are loaded once the
      // previous step's dV and dK are done.
      auto scores_other = [&](int it) -> bool {
        const uint32_t par = static_cast<uint32_t>(it) & 1u;
        if (!mbar_wait_warp(full + kQo, par, ab)) return false;
        tc_fence_after();
        scores(it, false, false, true);
        if (!mbar_wait_warp(full + kDo, par, ab)) return false;
        tc_fence_after();
        scores(it, true, false, true);
        mma_commit_warp(empty + kQo);
        mma_commit_warp(empty + kDo);
        return true;
      };
      auto scores_own = [&](int it) -> bool {
        const uint32_t par = static_cast<uint32_t>(it) & 1u;
        if (!mbar_wait_warp(full + kQh, par, ab)) return false;
        tc_fence_after();
        scores(it, false, true, false);
        if (!mbar_wait_warp(full + kDh, par, ab)) return false;
        tc_fence_after();
        scores(it, true, true, false);
#ifdef SDPA_TEST_WITHHOLD_FIRST_S_COMMIT
        // (test builds only, never in libsdpa.so: the first score tile is
        // never signalled, so the compute warps' bounded wait runs out and
        // every other role leaves through the abort flag or its own limit)
        if (it == 0) return true;
#endif
        mma_commit_warp(s_full);
        return true;
      };
      bool ok = mbar_wait_warp(kv_full, 0, ab);
      tc_fence_after();
      ok = ok && scores_other(0) && scores_own(0);
      for (int it = 0; ok && it < n_it; ++it) {
        const uint32_t par = static_cast<uint32_t>(it) & 1u;
        // the next step's scores over the other half's boxes go into the
        // other score buffer while the softmax works on this step's (that
        // buffer's last reader, the softmax of step it - 1, is done: its
        // P was waited for before step it - 1's products)
        if (it + 1 < n_it && !(ok = scores_other(it + 1))) break;
        // P^T and dS^T of step it are in shared memory
        ok = mbar_wait_warp(p_full, par, ab);
        if (!ok) break;
        tc_fence_after();
        const uint32_t bp = desc_lo(smem_base + kPOff, 16);
        const uint32_t bds = desc_lo(smem_base + kDsOff, 16);
        // dK first: its commit frees this half's Q part, the first of the
        // next step's own parts that the producer refills, while dV and dQ^T
        // run; dV's commit then frees the dO part
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const bool dv = g == 1;
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
            // 128 columns of d: boxes 2 mb, 2 mb + 1 of the own part, 4 KB apart
            const uint32_t a = desc_lo(smem_base + (dv ? kDohOff : kQhOff) + 2 * mb * kQBox, kQBox);
#pragma unroll
            for (int k = 0; k < kBN / 16; ++k) {
              const uint32_t ka = static_cast<uint32_t>(k * 16 * 128) >> 4;   // 16 query rows
              const uint32_t kb = static_cast<uint32_t>(k * 32) >> 4;         // 16 queries of a row
              mma_bf16_ss_warp(tmem + (dv ? kColDV : kColDK) + mb * 64, a + ka, kDescHi,
                               (dv ? bp : bds) + kb, kDescHi, kIdescG, (it > 0 || k > 0) ? 1u : 0u);
            }
          }
          mma_commit_warp(empty + (dv ? kDh : kQh));
        }
        // dQ^T(it) = K[:, half]^T dS^T(it) into buffer it & 1, once the
        // epilogue has read what step it - 2 left there
        const int b = it & 1;
        if (it >= 2) {
          ok = mbar_wait_warp(dq_empty + b, static_cast<uint32_t>((it - 2) >> 1) & 1u, ab);
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t bdq = desc_lo(smem_base + kDsOff, kKeys * 128);
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
          const uint32_t ak =
              desc_lo(smem_base + kKOff + (half * kHalfBoxes + 2 * mb) * kKVBox, kKVBox);
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k) {
            const uint32_t kk = static_cast<uint32_t>(k * 16 * 128) >> 4;   // 16 key rows
            mma_bf16_ss_warp(tmem + kColDQ + b * 64 + mb * 32, ak + kk, kDescHi, bdq + kk, kDescHi,
                             kIdescQ, k > 0 ? 1u : 0u);
          }
        }
        mma_commit_warp(dq_full + b);
        // this half's scores of the next step; its commit of s_full covers
        // this step's products, so the softmax may then overwrite P and dS
        if (it + 1 < n_it && !(ok = scores_own(it + 1))) break;
      }
      if (ok) mma_commit_warp(acc_full);
      mma_commit_warp(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= kEpilogueWarp0) {
    const int quarter = warp & 3;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* staging = reinterpret_cast<float*>(smem + kStagingOff + (warp - kEpilogueWarp0) * kStagingWarp);
    bool ok = true;
    // ---- dQ^T of each step: lanes are d, columns queries
    for (int j = 0; j < n_it; ++j) {
      const int b = j & 1;
      ok = mbar_wait_warp(dq_full + b, static_cast<uint32_t>(j >> 1) & 1u, ab);
      if (!ok) break;
      tc_fence_after();
      uint32_t g0[32], g1[32];
      tmem_ld32(lane_base + kColDQ + b * 64, g0);
      tmem_ld32(lane_base + kColDQ + b * 64 + 32, g1);
      tmem_ld_wait();
      reg_fence(g0);
      reg_fence(g1);
      tc_fence_before();
      mbar_arrive(dq_empty + b);
#pragma unroll
      for (int mb = 0; mb < 2; ++mb) {
        // the previous reduce has finished reading the staging tile
        if (lane == 0) tma_store_wait_read();
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 32; ++e) staging[e * 32 + lane] = __uint_as_float(mb ? g1[e] : g0[e]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&p.tm_dq, staging, half * 256 + mb * 128 + quarter * 32,
                            (i_lo + j) * kBN, bh);
          tma_store_commit();
        }
      }
    }
    // every reduce of this warp has completed (and read its staging tile)
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
    // ---- dV and dK (scaled): this warp's 32 columns of d in each 128-column
    // block, 64 key rows, transposed through its staging tile
    if (!__any_sync(0xffffffffu, *abort_flag != 0)) {
      bool have = ok && n_it > 0;
      if (have) {
        have = mbar_wait_warp(acc_full, 0, ab);
        tc_fence_after();
      }
      if (have || n_it == 0) {
        uint16_t* tile = reinterpret_cast<uint16_t*>(staging);   // [64 keys][32 d] bf16
#pragma unroll 1
        for (int t = 0; t < 4; ++t) {
          const int mb = t & 1;
          const bool is_k = t >= 2;
          const uint32_t col = (is_k ? kColDK : kColDV) + static_cast<uint32_t>(mb * 64);
          const float mul = is_k ? p.scale : 1.f;
          uint32_t a0[32], a1[32];
          if (have) {
            tmem_ld32(lane_base + col, a0);
            tmem_ld32(lane_base + col + 32, a1);
            tmem_ld_wait();
            reg_fence(a0);
            reg_fence(a1);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) a0[e] = a1[e] = 0u;
          }
          __syncwarp();   // the previous copy-out has read the tile
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const uint32_t v0 = pack_bf16x2(__uint_as_float(a0[e]) * mul, 0.f);
            const uint32_t v1 = pack_bf16x2(__uint_as_float(a1[e]) * mul, 0.f);
            tile[e * 32 + lane] = static_cast<uint16_t>(v0 & 0xffffu);
            tile[(32 + e) * 32 + lane] = static_cast<uint16_t>(v1 & 0xffffu);
          }
          __syncwarp();
          // 64 rows of 64 bytes: four 16-byte pieces per row
          uint16_t* dst = is_k ? p.dk : p.dv;
          const int col0 = half * 256 + mb * 128 + quarter * 32;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int piece = u * 32 + lane;
            const int row = piece >> 2, c = piece & 3;
            const int key = key0 + row;
            if (key < p.n_k) {
              const uint4 v = *reinterpret_cast<const uint4*>(tile + row * 32 + c * 8);
              *reinterpret_cast<uint4*>(dst + (static_cast<long long>(bh) * p.n_k + key) * kD + col0 +
                                        c * 8) = v;
            }
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------- compute warps
    // Lanes 16..31 read tensor-memory lanes that the M = 64 scores leave
    // unwritten; they compute on them but store nothing.
    const int quarter = warp & 3;
    const int qh = warp >> 2;                         // queries 16 qh .. +16 of each step
    const bool active = lane < 16;
    const int r = quarter * 16 + (lane & 15);         // key row of the tile
    const int key = key0 + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int it = 0; it < n_it; ++it) {
      const int b = it & 1;
      // the step's -lse2 and -D into registers while the scores still run
      const int vs = it % kVecSlots;
      if (!mbar_wait_warp(vec_full + vs, static_cast<uint32_t>(it / kVecSlots) & 1u, ab)) break;
      const uint32_t vec = smem_base + kVecOff + vs * kVecBytes + qh * 16 * 4;
      float4 nlv[4], ndv[4];
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4) {
        nlv[e4] = lds_f4(vec + e4 * 16);
        ndv[e4] = lds_f4(vec + kBN * 4 + e4 * 16);
      }
      if (!mbar_wait_warp(s_full, static_cast<uint32_t>(it) & 1u, ab)) break;
      tc_fence_after();
      const int q0 = (i_lo + it) * kBN + qh * 16;
      // this key sees all 16 queries: no per-element mask
      const bool all = !active || (key < kv_len && (!causal || key <= q0) &&
                                   key >= q0 + 15 - p.win_left && key <= q0 + p.win_right);
      uint32_t sv[16], dp[16];
      const uint32_t sbuf = static_cast<uint32_t>(b * 64);   // this step's score buffer
      tmem_ld16(lane_base + kColS + sbuf + qh * 16, sv);
      tmem_ld16(lane_base + kColDP + sbuf + qh * 16, dp);
      tmem_ld_wait();
      reg_fence(sv);
      reg_fence(dp);
      uint32_t pk[8], dk[8];
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
      auto rows = [&](auto masked) {
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          const float4 nl = nlv[e4];
          const float4 nd = ndv[e4];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = e4 * 4 + u * 2;
            const float2 nl2 = u ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y);
            const float2 nd2 = u ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y);
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                        sc2, nl2);
            float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
            if (decltype(masked)::value) {
              const int q = q0 + e;
              if (!(key < kv_len && (!causal || key <= q) && key >= q - p.win_left &&
                    key <= q + p.win_right))
                p0 = 0.f;
              if (!(key < kv_len && (!causal || key <= q + 1) && key >= q + 1 - p.win_left &&
                    key <= q + 1 + p.win_right))
                p1 = 0.f;
            }
            const float2 t = __fadd2_rn(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                        nd2);
            const float2 ds = __fmul2_rn(make_float2(p0, p1), t);
            pk[e >> 1] = pack_bf16x2(p0, p1);
            dk[e >> 1] = pack_bf16x2(ds.x, ds.y);
          }
        }
      };
      if (__all_sync(0xffffffffu, all))
        rows(std::false_type{});
      else
        rows(std::true_type{});
      // row r of P^T and dS^T, queries [16 qh, +16): 16-byte chunks 2 qh, 2 qh + 1
#pragma unroll
      for (int c = 0; c < 2 && active; ++c) {
        const uint32_t off = sw128_offset(static_cast<uint32_t>(r), static_cast<uint32_t>(qh * 2 + c));
        *reinterpret_cast<uint4*>(smem + kPOff + off) =
            make_uint4(pk[c * 4 + 0], pk[c * 4 + 1], pk[c * 4 + 2], pk[c * 4 + 3]);
        *reinterpret_cast<uint4*>(smem + kDsOff + off) =
            make_uint4(dk[c * 4 + 0], dk[c * 4 + 1], dk[c * 4 + 2], dk[c * 4 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace w512
}  // namespace

int bwd_key_tile(int d_k) { return d_k == w512::kD ? w512::kKeys : 128; }
int bwd_query_step(int d_k) { return d_k == w512::kD ? w512::kBN : 64; }

cudaError_t launch_sdpa_bwd_w512(const SdpaBwdParams& bp, bool after_prep, cudaStream_t stream) {
  const int smem = w512::kSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(w512::sdpa_bwd_tc_w512,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  const long long blocks = static_cast<long long>(bp.num_kv_tiles) * bp.b * bp.h * 2;
  if (blocks == 0) return cudaSuccess;
  return launch_kernel(w512::sdpa_bwd_tc_w512, dim3(static_cast<unsigned>(blocks)),
                       dim3(w512::kThreads), smem, stream, after_prep, bp);
}

}  // namespace sdpa
