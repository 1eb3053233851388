// Gradients of scaled dot-product attention for training ("Attention Is All
// You Need", section 5, applied to Eq. (1) of section 3.2.1).  With
// S = scale Q K^T, P = softmax(S) (masked entries 0), O = P V and upstream
// dO:
//   dV = P^T dO,  dP = dO V^T,  D_i = dO_i . O_i,  dS = P o (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
// P is recomputed from the forward's per-row log-sum-exp, never stored.
//
//   sdpa_bwd_prep        -D_i = -dO_i . O_i and the negated log-sum-exp in
//                        log2 units for every query row (padded to whole
//                        128-row tiles with 0 and -inf, so padded rows get
//                        P = 0); zeroes the fp32 dQ accumulator.
//   sdpa_bwd_tc_n64<DK, DV>
//                        one CTA per (128-key tile, batch, head), walking in
//                        steps of 64 the queries that can see its keys; dK
//                        and dV accumulate in tensor memory, dQ leaves each
//                        step as a bulk reduce-add into the accumulator.
//   sdpa_bwd_dq_convert  dQ = scale * accumulator, rounded to bf16.
//
// Everything runs in the transposed frame, with the keys of the CTA in
// tensor-memory lanes.  The five products per step are
// S^T = K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q and dQ^T = K^T dS^T.
#include <cmath>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {
namespace {

// ------------------------------------------------------------------------
// 64-query steps with S^T / dP^T double-buffered in tensor memory, so the
// tensor core computes the next step's products while the compute warps turn
// the current ones into P^T and dS^T.
//   warps 0-7    compute: warp w serves key lanes 32 (w % 4) .. +32 and
//                query half w / 4 (32 queries) of each step; at the end they
//                write dK and dV.
//   warp 8       TMA producer (K_j, V_j once; Q_i, dO_i, lse2, D in 3 stages).
//   warp 9       MMA issuer (the whole warp; one elected lane issues each
//                instruction), in the order S(i+1), dP(i+1), dV(i), dK(i), dQ^T.
//   warps 10-13  dQ^T out of tensor memory into the staging tile.
// Tensor memory: buffer b = step & 1 holds S^T at 128 b (64 columns; P^T in
// bf16 over columns 128 b + 32 h .. +16 of each half h) and dP^T at
// 128 b + 64 (dS^T in bf16 the same way), dV at 256, dK at 256 + d_v.
// dQ^T = K^T dS^T (keyed by d):
//   d_k + d_v > 128: one N = 64 product per step into the dP^T half of its
//                buffer, drained through a 64 x d_k fp32 staging tile;
//   d_k + d_v <= 128: one N = 128 product per pair of steps into columns
//                384 .. 511, drained through a 128 x d_k staging tile.
// Each 64 rows then go into the fp32 dQ accumulator by one bulk reduce-add.
namespace n64 {

constexpr int kBM = 128;                 // keys per CTA
constexpr int kBN = 64;                  // queries per step
constexpr int kStages = 3;
constexpr int kThreads = 448;
constexpr int kCompute = 256;            // warps 0-7
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kEpilogueWarp0 = 10;       // warps 10-13: dQ^T out of tensor memory
constexpr int kEpilogue = 128;
constexpr int kHeadGroup = 4;            // heads whose key tiles run together
constexpr int kDsTile = kBM * kBN * 2;   // dS^T: 128 keys x 64 queries bf16 (128-byte rows)
constexpr int kVecBytes = 2 * kBN * 4;   // -lse2 and -D of one step
// kv_full, q_full[3], q_empty[3], s_full[2], p_full[2], dq_full[2],
// dq_empty[2], acc_full, drain, then (wide heads) part_full[4],
// part_empty[4], vec_full[3]
constexpr int kNumBars = 1 + 2 * kStages + 8 + 2 + 11;
constexpr uint32_t kIdescS = idesc_bf16(kBM, kBN, false, false);   // S^T, dP^T
// dQ^T = K^T dS^T always with M = 128 lanes of d: for d_k < 128 the upper lanes
// read the tiles that follow K in shared memory and are discarded.
constexpr uint32_t kIdescQ = idesc_bf16(128, kBN, true, true);
constexpr uint32_t kIdescQ2 = idesc_bf16(128, 2 * kBN, true, true);   // a pair of steps
// dS^T rows are 128 bytes (64 queries): 128-byte swizzle, 8-row groups 1024 apart
constexpr uint32_t kDsHi = (1024u >> 4) | (1u << 14) | (2u << 29);

// Layout of an operand whose rows hold D bf16 values (K and Q at d_k; V and
// dO at d_v): boxes of kBoxCols columns, rows of kRowBytes swizzled at that
// width (128-, 64- or 32-byte swizzle for d >= 64, 32, 16).
template <int D>
struct Lay {
  static constexpr int kBoxCols = D < 64 ? D : 64;
  static constexpr int kRowBytes = kBoxCols * 2;
  static constexpr uint32_t kLayout = kRowBytes == 128 ? 2u : (kRowBytes == 64 ? 4u : 6u);
  static constexpr uint32_t kSBO = 8 * kRowBytes;
  static constexpr int kStepsPerRow = kRowBytes / 32;       // K=16 steps per swizzled row
  static constexpr uint32_t kDescHi = (kSBO >> 4) | (1u << 14) | (kLayout << 29);
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kKVBox = 128 * kRowBytes;            // kBoxCols x 128 keys
  static constexpr int kQBox = 64 * kRowBytes;              // kBoxCols x 64 queries
  static constexpr int kKVTile = kBoxes * kKVBox;
  static constexpr int kQTile = kBoxes * kQBox;
  static_assert(kQBox % 1024 == 0 && kKVBox % 1024 == 0, "align");
};

// Shared memory and tensor memory of one CTA for key size DK and value
// size DV.  Tensor memory: the two score buffers (256 columns), dV at 256
// (DV columns), dK at 256 + DV (DK columns).  When DK + DV <= 128 the last
// 128 columns are free: dQ^T then goes there, one product of N = 128 per
// pair of query steps (four dS^T buffers, so that a pair's two are
// adjacent) instead of one N = 64 product per step into the dP^T half.
template <int DK, int DV>
struct Cfg {
  using LK = Lay<DK>;
  using LV = Lay<DV>;
  static constexpr bool kPairDq = DK + DV <= 128;
  // Heads wider than 128 (d_k = d_v = 256): dK, dV and dQ in 128-column
  // chunks, one CTA per chunk, each recomputing S^T and dP^T over the whole
  // head.  K and V stay resident (128 KB), which leaves room for one stage
  // of Q and dO and one dS^T buffer.  The stage's boxes come in four parts
  // with barriers of their own: Q's and dO's boxes of the other chunk, free
  // once the step's scores have read them, and this CTA's chunk of Q, free
  // once dK has read it, and of dO, once dV has; so the next step's loads
  // run while this step's softmax and products do.
  static constexpr bool kWide = DK > 128;
  static constexpr int kColsK = kWide ? 128 : DK;           // dK / dQ columns of a CTA
  static constexpr int kColsV = kWide ? 128 : DV;           // dV columns of a CTA
  static constexpr int kChunks = kWide ? DK / 128 : 1;      // CTAs per key tile
  static constexpr int kStagesQ = kWide ? 1 : kStages;      // Q / dO stages
  static constexpr int kDsBufs = kPairDq ? 4 : (kWide ? 1 : 2);
  // staged dQ rows per epilogue warp (the wide heads stage 32 query rows at a time)
  static constexpr int kDqRows = kPairDq ? 2 * kBN : (kWide ? 32 : kBN);
  static constexpr uint32_t kDqCol = 384;                   // paired dQ^T: 128 columns
  static constexpr int kDCols = DK < 32 ? DK : 32;          // dQ columns per epilogue warp
  static constexpr int kKOff = 0;
  static constexpr int kVOff = LK::kKVTile;
  static constexpr int kStageOff = kVOff + LV::kKVTile;     // Q then dO, per stage
  static constexpr int kStageBytes = LK::kQTile + LV::kQTile;
  static constexpr int kDsOff = kStageOff + kStagesQ * kStageBytes;   // dS^T buffers
  static constexpr int kStagingOff = kDsOff + kDsBufs * kDsTile;  // 4 warps x [kDqRows][kDCols] fp32
  static constexpr int kVecOff = kStagingOff + 4 * kDqRows * kDCols * 4;
  static constexpr int kVecBufs = kWide ? 3 : kStagesQ;       // -lse2 / -D slots
  static_assert(!kWide || kVecBufs == 3, "three vec_full barriers");
  static constexpr int kBarOff = kVecOff + kVecBufs * kVecBytes;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  static constexpr uint32_t kIdescDV = idesc_bf16(kBM, kColsV, false, true);  // dV (A in TMEM)
  static constexpr uint32_t kIdescDK = idesc_bf16(kBM, kColsK, false, true);  // dK (A in TMEM)
  static constexpr uint32_t kDkCol = 256 + kColsV;
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kStageOff % 1024 == 0 && kDsOff % 1024 == 0 && kStagingOff % 1024 == 0, "align");
  static_assert(kDkCol + kColsK <= (kPairDq ? kDqCol : 512u), "tensor memory");
  static_assert(!kWide || (DK == DV && DK % 128 == 0), "wide heads: equal sizes, 128-column chunks");
  // dQ^T's 128 lanes read 128 / kBoxCols boxes from K onward: all inside the CTA's memory
  static_assert((128 / LK::kBoxCols) * LK::kKVBox <= kBarOff, "dQ^T reads in bounds");
};

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1) sdpa_bwd_tc_n64(const __grid_constant__ SdpaBwdParams p) {
  using C = Cfg<DK, DV>;
  using LK = typename C::LK;
  using LV = typename C::LV;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t smem_base = smem_u32(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* kv_full = bar;
  uint64_t* q_full = bar + 1;
  uint64_t* q_empty = q_full + kStages;
  uint64_t* s_full = q_empty + kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* dq_full = p_full + 2;
  uint64_t* dq_empty = dq_full + 2;
  uint64_t* acc_full = dq_empty + 2;
  uint64_t* drain = acc_full + 1;
  // wide heads: parts 0..3 = Q other, dO other, Q own, dO own (box pairs)
  uint64_t* part_full = drain + 1;
  uint64_t* part_empty = part_full + 4;
  uint64_t* vec_full = part_empty + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(vec_full + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const AbortState ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh_count = p.b * p.h;
  // Column chunk of dK, dV and dQ (wide heads; else 0), then heads in groups
  // of kHeadGroup, each group's key tiles in ascending order (the longest
  // causal walks first): the dQ accumulator and the Q / dO rows of the heads
  // in flight stay in L2.
  const int chunk = static_cast<int>(blockIdx.x) % C::kChunks;
  const int idx = static_cast<int>(blockIdx.x) / C::kChunks;
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
  // Read before griddep_wait(): the lengths are the caller's input, which the
  // prep kernel this one may depend on never writes.
  int kv_len = p.n_k;
  if ((p.mask_kind & 2) && p.kv_lengths != nullptr) {
    kv_len = p.kv_lengths[bi];
    kv_len = kv_len < 0 ? 0 : (kv_len > p.n_k ? p.n_k : kv_len);
  }
  const int key0 = jt * kBM;
  const int2 qr = bwd_query_steps<kBM, kBN>(p, key0, kv_len);
  const int i_lo = qr.x, n_it = qr.y - qr.x;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(q_full + s, 1);
      mbar_init(q_empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, kCompute);
      mbar_init(dq_full + b, 1);
      mbar_init(dq_empty + b, kEpilogue);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(part_full + s, 1);
      mbar_init(part_empty + s, 1);
    }
    for (int s = 0; s < 3; ++s) mbar_init(vec_full + s, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every CTA holds its tensor memory now: the convert kernel may launch;
  // the prep kernel's vectors and zeroed accumulator must be complete.
  griddep_launch_dependents();
  griddep_wait();

  if (warp == kProducerWarp) {
    if (lane == 0 && n_it > 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      mbar_arrive_expect_tx(kv_full, LK::kKVTile + LV::kKVTile);
      for (int c = 0; c < LK::kBoxes; ++c)
        tma_load_4d(&p.tm_k, kv_full, smem + C::kKOff + c * LK::kKVBox, c * LK::kBoxCols, key0, hi, bi);
      for (int c = 0; c < LV::kBoxes; ++c)
        tma_load_4d(&p.tm_v, kv_full, smem + C::kVOff + c * LV::kKVBox, c * LV::kBoxCols, key0, hi, bi);
      if constexpr (C::kWide) {
        // four parts of two boxes each, in the order the MMA warp frees them:
        // Q other, dO other (after the step's scores over them), Q own (after
        // dK), dO own (after dV); the step's vectors go with the first part,
        // into one of three slots (the slot's last reader, the softmax of
        // step it - 3, finished before the scores of step it - 1 over the
        // other chunk were issued, and those freed this part)
        int issued[4] = {0, 0, 0, 0};
        int vec_issued = 0;
        bool go = true;
        uint8_t* st = smem + C::kStageOff;
        for (int it = 0; go && it < n_it; ++it) {
          const int q0 = (i_lo + it) * kBN;
#pragma unroll
          for (int pt = 0; pt < 4; ++pt) {
            if (it > 0 && !mbar_wait(part_empty + pt, static_cast<uint32_t>(it - 1) & 1u, ab)) {
              go = false;
              break;
            }
            const bool is_do = (pt & 1) != 0;
            const int c0 = 2 * (pt >= 2 ? chunk : 1 - chunk);
            mbar_arrive_expect_tx(part_full + pt, 2 * LK::kQBox);
            for (int j = 0; j < 2; ++j) {
              const int c = c0 + j;
              if (is_do)
                tma_load_4d(&p.tm_do, part_full + pt, st + LK::kQTile + c * LV::kQBox,
                            c * LV::kBoxCols, q0, hi, bi);
              else
                tma_load_4d(&p.tm_q, part_full + pt, st + c * LK::kQBox, c * LK::kBoxCols, q0, hi,
                            bi);
            }
            issued[pt] = it + 1;
            if (pt == 0) {
              uint64_t* vb = vec_full + it % C::kVecBufs;
              const long long vrow = static_cast<long long>(bh) * p.n_q_pad + q0;
              uint8_t* vec = smem + C::kVecOff + (it % C::kVecBufs) * kVecBytes;
              mbar_arrive_expect_tx(vb, kVecBytes);
              tma_load_1d(vec, p.neg_lse2 + vrow, kBN * 4, vb);
              tma_load_1d(vec + kBN * 4, p.neg_dvec + vrow, kBN * 4, vb);
              vec_issued = it + 1;
            }
          }
        }
        // let the copies still in flight land before the CTA can exit
        mbar_wait_drain(kv_full, 0);
        for (int pt = 0; pt < 4; ++pt)
          if (issued[pt] > 0)
            mbar_wait_drain(part_full + pt, static_cast<uint32_t>(issued[pt] - 1) & 1u);
        for (int it = max(0, vec_issued - C::kVecBufs); it < vec_issued; ++it)
          mbar_wait_drain(vec_full + it % C::kVecBufs, static_cast<uint32_t>(it / C::kVecBufs) & 1u);
      } else {
      int issued = 0;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % C::kStagesQ;
        const uint32_t use = static_cast<uint32_t>(it / C::kStagesQ);
        if (it >= C::kStagesQ && !mbar_wait(q_empty + s, (use - 1) & 1u, ab)) break;
        uint8_t* st = smem + C::kStageOff + s * C::kStageBytes;
        const int q0 = (i_lo + it) * kBN;
        mbar_arrive_expect_tx(q_full + s, C::kStageBytes + kVecBytes);
        for (int c = 0; c < LK::kBoxes; ++c)
          tma_load_4d(&p.tm_q, q_full + s, st + c * LK::kQBox, c * LK::kBoxCols, q0, hi, bi);
        for (int c = 0; c < LV::kBoxes; ++c)
          tma_load_4d(&p.tm_do, q_full + s, st + LK::kQTile + c * LV::kQBox, c * LV::kBoxCols, q0,
                      hi, bi);
        const long long vrow = static_cast<long long>(bh) * p.n_q_pad + q0;
        uint8_t* vec = smem + C::kVecOff + s * kVecBytes;
        tma_load_1d(vec, p.neg_lse2 + vrow, kBN * 4, q_full + s);
        tma_load_1d(vec + kBN * 4, p.neg_dvec + vrow, kBN * 4, q_full + s);
        issued = it + 1;
      }
      mbar_wait_drain(kv_full, 0);
      for (int it = max(0, issued - C::kStagesQ); it < issued; ++it)
        mbar_wait_drain(q_full + it % C::kStagesQ, static_cast<uint32_t>(it / C::kStagesQ) & 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    // The whole warp runs this loop in step (warp-uniform waits and
    // descriptors); one elected lane issues every product and commit.
    if (n_it > 0) {
      const uint32_t k_smem = smem_base + C::kKOff;
      const uint32_t v_smem = smem_base + C::kVOff;
      // Shared-memory descriptors as 32-bit halves: every operand here is
      // 128-byte swizzled with 8-row groups 1024 bytes apart, so the high
      // half is one constant and a k step only adds to the start address.
      auto lo = [](uint32_t addr, uint32_t lbo) { return (addr >> 4) | ((lbo >> 4) << 16); };
      // S^T(it) = K_j Q_i^T (dp false) or dP^T(it) = V_j dO_i^T (dp true) into buffer it & 1
      auto issue_s = [&](int it, bool dp) {
        const uint32_t st = smem_base + C::kStageOff + (it % C::kStagesQ) * C::kStageBytes;
        const uint32_t d = tmem + static_cast<uint32_t>((it & 1) * 128 + (dp ? 64 : 0));
        auto product = [&](auto lay, uint32_t a_addr, uint32_t b_addr, int dsize) {
          using L = decltype(lay);
          const uint32_t a0 = lo(a_addr, 16), b0 = lo(b_addr, 16);
#pragma unroll
          for (int k = 0; k < dsize / 16; ++k) {
            constexpr int kS = L::kStepsPerRow;
            mma_bf16_ss_warp(d, a0 + static_cast<uint32_t>(((k / kS) * L::kKVBox + (k % kS) * 32) >> 4),
                             L::kDescHi,
                             b0 + static_cast<uint32_t>(((k / kS) * L::kQBox + (k % kS) * 32) >> 4),
                             L::kDescHi, kIdescS, k > 0 ? 1u : 0u);
          }
        };
        if (dp)
          product(LV{}, v_smem, st + LK::kQTile, DV);
        else
          product(LK{}, k_smem, st, DK);
      };
      // Wide heads: S^T(it) and dP^T(it) part by part as the stage's parts
      // land.  wide_scores_other issues them over the other chunk's boxes and
      // frees those two parts; wide_scores_own adds this chunk's boxes and
      // commits s_full.  dP^T(it) lands where dQ^T(it - 2) was, so it waits
      // for that step's epilogue.
      auto wide_part = [&](int it, bool dp, bool own, bool first) {
        const uint32_t st = smem_base + C::kStageOff;
        const int c0 = 2 * (own ? chunk : 1 - chunk);
        const uint32_t d = tmem + static_cast<uint32_t>((it & 1) * 128 + (dp ? 64 : 0));
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = c0 + j;
          const uint32_t a0 = lo((dp ? v_smem : k_smem) + c * LK::kKVBox, 16);
          const uint32_t b0 = lo(st + (dp ? LK::kQTile : 0) + c * LK::kQBox, 16);
#pragma unroll
          for (int kk = 0; kk < LK::kStepsPerRow; ++kk)
            mma_bf16_ss_warp(d, a0 + static_cast<uint32_t>(kk * 2), LK::kDescHi,
                             b0 + static_cast<uint32_t>(kk * 2), LK::kDescHi, kIdescS,
                             (first && j == 0 && kk == 0) ? 0u : 1u);
        }
      };
      auto wide_scores_other = [&](int it) -> bool {
        const uint32_t par = static_cast<uint32_t>(it) & 1u;
        if (!mbar_wait_warp(part_full + 0, par, ab)) return false;
        tc_fence_after();
        wide_part(it, false, false, true);
        if (it >= 2) {
          if (!mbar_wait_warp(dq_empty + (it & 1), static_cast<uint32_t>((it - 2) >> 1) & 1u, ab))
            return false;
          tc_fence_after();
        }
        if (!mbar_wait_warp(part_full + 1, par, ab)) return false;
        tc_fence_after();
        wide_part(it, true, false, true);
        mma_commit_warp(part_empty + 0);
        mma_commit_warp(part_empty + 1);
        return true;
      };
      auto wide_scores_own = [&](int it) -> bool {
        const uint32_t par = static_cast<uint32_t>(it) & 1u;
        if (!mbar_wait_warp(part_full + 2, par, ab)) return false;
        tc_fence_after();
        wide_part(it, false, true, false);
        if (!mbar_wait_warp(part_full + 3, par, ab)) return false;
        tc_fence_after();
        wide_part(it, true, true, false);
#ifdef SDPA_TEST_WITHHOLD_FIRST_S_COMMIT
        if (it == 0) return true;
#endif
        mma_commit_warp(s_full + (it & 1));
        return true;
      };
      bool ok = mbar_wait_warp(kv_full, 0, ab);
      if constexpr (C::kWide) {
        tc_fence_after();
        ok = ok && wide_scores_other(0) && wide_scores_own(0);
      } else {
        ok = ok && mbar_wait_warp(q_full, 0, ab);
        tc_fence_after();
        if (ok) {
          issue_s(0, false);
          issue_s(0, true);
#ifndef SDPA_TEST_WITHHOLD_FIRST_S_COMMIT
          mma_commit_warp(s_full);
#endif
          // (test builds only, never in libsdpa.so: the first S^T / dP^T tile
          // is never signalled, so the compute warps' bounded wait runs out and
          // every other role leaves through the abort flag or its own limit)
        }
      }
      if constexpr (C::kWide) {
        // This CTA's chunk of dV, dK and dQ^T reads the matching 128 columns
        // (two boxes) of dO, Q and K.
        const uint32_t col_boxes = static_cast<uint32_t>(chunk * (128 / LK::kBoxCols));
        for (int it = 0; ok && it < n_it; ++it) {
          const int b = it & 1;
          // the next step's scores over the other chunk's boxes go into the
          // other buffer while the compute warps work on this step's
          if (it + 1 < n_it && !(ok = wide_scores_other(it + 1))) break;
          ok = mbar_wait_warp(p_full + b, static_cast<uint32_t>(it >> 1) & 1u, ab);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = smem_base + C::kStageOff;
          const uint32_t buf = tmem + static_cast<uint32_t>(b * 128);
          const uint32_t bdo = lo(st + LK::kQTile + col_boxes * LV::kQBox, LV::kQBox);
          const uint32_t bq = lo(st + col_boxes * LK::kQBox, LK::kQBox);
          // dK first: its commit frees this chunk's Q boxes, the first own
          // part the producer refills, while dV and dQ^T run; dV's commit
          // then frees the dO boxes
#pragma unroll
          for (int k = 0; k < kBN / 16; ++k) {
            const uint32_t col = static_cast<uint32_t>((k >> 1) * 32 + (k & 1) * 8);
            mma_bf16_ts_warp(tmem + C::kDkCol, buf + 64 + col,
                             bq + (static_cast<uint32_t>(k * 16 * LK::kRowBytes) >> 4), LK::kDescHi,
                             C::kIdescDK, (it > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit_warp(part_empty + 2);
#pragma unroll
          for (int k = 0; k < kBN / 16; ++k) {
            const uint32_t col = static_cast<uint32_t>((k >> 1) * 32 + (k & 1) * 8);
            mma_bf16_ts_warp(tmem + 256, buf + col,
                             bdo + (static_cast<uint32_t>(k * 16 * LV::kRowBytes) >> 4), LV::kDescHi,
                             C::kIdescDV, (it > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit_warp(part_empty + 3);
          // dQ^T(it) = K_j[:, chunk]^T dS^T(it) into the dP^T half of buffer b
          // (dP^T(it) is consumed: the compute warps released P(it))
          const uint32_t ak = lo(smem_base + C::kKOff + col_boxes * LK::kKVBox, LK::kKVBox);
          const uint32_t bds = lo(smem_base + C::kDsOff, kDsTile);
#pragma unroll
          for (int k = 0; k < kBM / 16; ++k) {
            const uint32_t ka = static_cast<uint32_t>(k * 16 * LK::kRowBytes) >> 4;
            const uint32_t kb = static_cast<uint32_t>(k * 16 * 128) >> 4;
            mma_bf16_ss_warp(buf + 64, ak + ka, LK::kDescHi, bds + kb, kDsHi, kIdescQ,
                             k > 0 ? 1u : 0u);
          }
          mma_commit_warp(dq_full + b);
          if (it + 1 < n_it && !(ok = wide_scores_own(it + 1))) break;
        }
      }
      for (int it = 0; !C::kWide && ok && it < n_it; ++it) {
        const int b = it & 1;
        if (it + 1 < n_it) {
          const int nx = it + 1;
          ok = mbar_wait_warp(q_full + nx % kStages, static_cast<uint32_t>(nx / kStages) & 1u, ab);
          if (!ok) break;
          tc_fence_after();
          issue_s(nx, false);
          // dP^T(it+1) lands where dQ^T(it-1) was: its epilogue must have read it
          // (paired dQ^T has columns of its own)
          if (!C::kPairDq && it >= 1) {
            ok = mbar_wait_warp(dq_empty + (nx & 1), static_cast<uint32_t>((it - 1) >> 1) & 1u, ab);
            if (!ok) break;
            tc_fence_after();
          }
          issue_s(nx, true);
          mma_commit_warp(s_full + (nx & 1));
        }
        ok = mbar_wait_warp(p_full + b, static_cast<uint32_t>(it >> 1) & 1u, ab);
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = smem_base + C::kStageOff + (it % kStages) * C::kStageBytes;
        const uint32_t buf = tmem + static_cast<uint32_t>(b * 128);
        // dV += P^T dO_i, dK += dS^T Q_i: 16 queries per step; queries
        // [32h, 32h+32) sit in columns 32h .. 32h+16 of the S^T / dP^T halves
        const uint32_t bdo = lo(st + LK::kQTile, LV::kQBox), bq = lo(st, LK::kQBox);
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k) {
          const uint32_t col = static_cast<uint32_t>((k >> 1) * 32 + (k & 1) * 8);
          mma_bf16_ts_warp(tmem + 256, buf + col,
                           bdo + (static_cast<uint32_t>(k * 16 * LV::kRowBytes) >> 4), LV::kDescHi,
                           C::kIdescDV, (it > 0 || k > 0) ? 1u : 0u);
          mma_bf16_ts_warp(tmem + C::kDkCol, buf + 64 + col,
                           bq + (static_cast<uint32_t>(k * 16 * LK::kRowBytes) >> 4), LK::kDescHi,
                           C::kIdescDK, (it > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit_warp(q_empty + it % kStages);
        const uint32_t ak = lo(k_smem, LK::kKVBox);
        if constexpr (C::kPairDq) {
          // dQ^T of steps (it-1, it) at odd it, or of a last step alone:
          // K_j^T [dS^T(it-1) | dS^T(it)] into columns kDqCol .. +128
          const bool last = it + 1 == n_it;
          if ((it & 1) || last) {
            const int grp = it >> 1;
            if (grp >= 1) {
              ok = mbar_wait_warp(dq_empty, static_cast<uint32_t>(grp - 1) & 1u, ab);
              if (!ok) break;
              tc_fence_after();
            }
            const int first = (it & 1) ? it - 1 : it;
            const uint32_t bds = lo(smem_base + C::kDsOff + (first & 3) * kDsTile, kDsTile);
            const uint32_t idq = (it & 1) ? kIdescQ2 : kIdescQ;
#pragma unroll
            for (int k = 0; k < kBM / 16; ++k) {
              const uint32_t ka = static_cast<uint32_t>(k * 16 * LK::kRowBytes) >> 4;
              const uint32_t kb = static_cast<uint32_t>(k * 16 * 128) >> 4;
              mma_bf16_ss_warp(tmem + C::kDqCol, ak + ka, LK::kDescHi, bds + kb, kDsHi, idq,
                               k > 0 ? 1u : 0u);
            }
            mma_commit_warp(dq_full);
          }
        } else {
          // dQ^T(it) = K_j^T dS^T(it): 16 keys per step, into the dP^T half of buffer b
          const uint32_t bds = lo(smem_base + C::kDsOff + b * kDsTile, kDsTile);
#pragma unroll
          for (int k = 0; k < kBM / 16; ++k) {
            const uint32_t ka = static_cast<uint32_t>(k * 16 * LK::kRowBytes) >> 4;  // 16 key rows of K
            const uint32_t kb = static_cast<uint32_t>(k * 16 * 128) >> 4;            // of dS^T
            mma_bf16_ss_warp(buf + 64, ak + ka, LK::kDescHi, bds + kb, kDsHi, kIdescQ,
                             k > 0 ? 1u : 0u);
          }
          mma_commit_warp(dq_full + b);
        }
      }
      if (ok) mma_commit_warp(acc_full);
      mma_commit_warp(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= kEpilogueWarp0) {
    // ------------------------------------------ dQ^T out of tensor memory
    // Warp 10 + k serves the d lanes 32 q .. +32 (q = warp % 4) of every
    // step.  It writes its [64 queries][32 d] block into its own staging
    // tile and adds that block into the fp32 accumulator with one tensor
    // reduce; rows past n_q are clipped by the copy engine.
    const int quarter = warp & 3;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* staging = reinterpret_cast<float*>(smem + C::kStagingOff) + quarter * (C::kDqRows * C::kDCols);
    const bool active = quarter * 32 < DK;   // lanes 32 q .. are d values only below d_k
    // Stages 64 query rows (two 32-column TMEM loads from `col`) at row `row0`
    // of this warp's staging tile.
    auto load_half = [&](uint32_t col, uint32_t (&g0)[32], uint32_t (&g1)[32]) {
      tmem_ld32(lane_base + col, g0);
      tmem_ld32(lane_base + col + 32, g1);
      tmem_ld_wait();
      reg_fence(g0);
      reg_fence(g1);
    };
    auto stage_half = [&](int row0, const uint32_t (&g0)[32], const uint32_t (&g1)[32]) {
      if (lane < C::kDCols) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          staging[(row0 + e) * C::kDCols + lane] = __uint_as_float(g0[e]);
          staging[(row0 + 32 + e) * C::kDCols + lane] = __uint_as_float(g1[e]);
        }
      }
    };
    if constexpr (C::kPairDq) {
      // one group per pair of steps (the last may be a single step)
      for (int grp = 0; 2 * grp < n_it; ++grp) {
        const bool two = 2 * grp + 1 < n_it;
        if (!mbar_wait_warp(dq_full, static_cast<uint32_t>(grp) & 1u, ab)) break;
        tc_fence_after();
        uint32_t g0[32], g1[32];
        load_half(C::kDqCol, g0, g1);
        if (active) {
          // this warp's previous reduces have finished reading the staging tile
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          __syncwarp();
          stage_half(0, g0, g1);
        }
        if (two) {
          load_half(C::kDqCol + 64, g0, g1);
          if (active) stage_half(kBN, g0, g1);
        }
        tc_fence_before();
        mbar_arrive(dq_empty);
        if (!active) continue;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&p.tm_dq, staging, quarter * 32, (i_lo + 2 * grp) * kBN, bh);
          if (two)
            tma_reduce_add_3d(&p.tm_dq, staging + kBN * C::kDCols, quarter * 32,
                              (i_lo + 2 * grp + 1) * kBN, bh);
          tma_store_commit();
        }
      }
    } else if constexpr (C::kWide) {
      // 64 query rows of this warp's 32 d columns (of the CTA's chunk), staged
      // and reduced 32 rows at a time
      for (int j = 0; j < n_it; ++j) {
        const int b = j & 1;
        if (!mbar_wait_warp(dq_full + b, static_cast<uint32_t>(j >> 1) & 1u, ab)) break;
        tc_fence_after();
        uint32_t g0[32], g1[32];
        load_half(static_cast<uint32_t>(b * 128 + 64), g0, g1);
        tc_fence_before();
        mbar_arrive(dq_empty + b);
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          // this warp's previous reduce has finished reading the staging tile
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          __syncwarp();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            staging[e * C::kDCols + lane] = __uint_as_float(hq ? g1[e] : g0[e]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&p.tm_dq, staging, chunk * 128 + quarter * 32,
                              (i_lo + j) * kBN + hq * 32, bh);
            tma_store_commit();
          }
        }
      }
    } else {
      for (int j = 0; j < n_it; ++j) {
        const int b = j & 1;
        if (!mbar_wait_warp(dq_full + b, static_cast<uint32_t>(j >> 1) & 1u, ab)) break;
        tc_fence_after();
        uint32_t g0[32], g1[32];
        load_half(static_cast<uint32_t>(b * 128 + 64), g0, g1);
        tc_fence_before();
        mbar_arrive(dq_empty + b);
        if (!active) continue;
        // this warp's previous reduce has finished reading the staging tile
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
        stage_half(0, g0, g1);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&p.tm_dq, staging, quarter * 32, (i_lo + j) * kBN, bh);
          tma_store_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();   // this warp's last reduce has finished
  } else {
    // ------------------------------------------------------- compute warps
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int r = quarter * 32 + lane;                // key lane
    const int key = key0 + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true;

    for (int it = 0; it < n_it; ++it) {
      const int b = it & 1;
      // the step's -lse2 and -D: with the stage (narrow heads) or in a slot
      // of their own (wide heads, whose stage parts are refilled early)
      const int s = it % (C::kWide ? C::kVecBufs : C::kStagesQ);
      if constexpr (C::kWide)
        ok = mbar_wait_warp(vec_full + s, static_cast<uint32_t>(it / C::kVecBufs) & 1u, ab);
      else
        ok = mbar_wait_warp(q_full + s, static_cast<uint32_t>(it / C::kStagesQ) & 1u, ab);
      ok = ok && mbar_wait_warp(s_full + b, static_cast<uint32_t>(it >> 1) & 1u, ab);
      if (!ok) break;
      tc_fence_after();
      const int qh0 = (i_lo + it) * kBN + half * 32;
      // -lse2 and -D of this half's 32 queries (broadcast shared loads)
      const uint32_t vec = smem_base + C::kVecOff + s * kVecBytes + half * 32 * 4;
      // this key sees every query of its half: no per-element mask
      const bool full = key < kv_len && (!causal || key <= qh0) && key >= qh0 + 31 - p.win_left &&
                        key <= qh0 + p.win_right;
      const uint32_t s_col = static_cast<uint32_t>(b * 128 + half * 32);
      uint32_t sv[32], dp[32];
      tmem_ld32(lane_base + s_col, sv);
      tmem_ld32(lane_base + s_col + 64, dp);
      tmem_ld_wait();
      reg_fence(sv);
      reg_fence(dp);
      uint32_t pk[16], dk[16];
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
      // P^T = exp2(S^T scale log2e - lse2), dS^T = P^T (dP^T - D), two at a time
      auto rows = [&](auto masked) {
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 nl = lds_f4(vec + e4 * 16);
          const float4 nd = lds_f4(vec + kBN * 4 + e4 * 16);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = e4 * 4 + u * 2;
            const float2 nl2 = u ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y);
            const float2 nd2 = u ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y);
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                        sc2, nl2);
            float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
            if (decltype(masked)::value) {
              const int q = qh0 + e;
              if (!(key < kv_len && (!causal || key <= q) && key >= q - p.win_left &&
                    key <= q + p.win_right))
                p0 = 0.f;
              if (!(key < kv_len && (!causal || key <= q + 1) && key >= q + 1 - p.win_left &&
                    key <= q + 1 + p.win_right))
                p1 = 0.f;
            }
            const float2 t = __fadd2_rn(
                make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd2);
            const float2 ds = __fmul2_rn(make_float2(p0, p1), t);
            pk[e >> 1] = pack_bf16x2(p0, p1);
            dk[e >> 1] = pack_bf16x2(ds.x, ds.y);
          }
        }
      };
      if (__all_sync(0xffffffffu, full))
        rows(std::false_type{});
      else
        rows(std::true_type{});
      tmem_st16(lane_base + s_col, pk);
      tmem_st16(lane_base + s_col + 64, dk);
      // dS^T row r, queries [32 half, +32): 16-byte chunks 4 half .. +4 of the 128-byte row
      uint8_t* dsb = smem + C::kDsOff + (it & (C::kDsBufs - 1)) * kDsTile;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v = make_uint4(dk[c * 4 + 0], dk[c * 4 + 1], dk[c * 4 + 2], dk[c * 4 + 3]);
        *reinterpret_cast<uint4*>(dsb + sw128_offset(static_cast<uint32_t>(r),
                                                     static_cast<uint32_t>(half * 4 + c))) = v;
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full + b);
    }
    // ---- dK (scaled) and dV rows: warp half h takes the half h of each tensor's columns
    if (!__any_sync(0xffffffffu, *abort_flag != 0)) {
      bool have = ok && n_it > 0;
      if (have) {
        have = mbar_wait_warp(acc_full, 0, ab);
        tc_fence_after();
      }
      if (have || n_it == 0) {
        // one tensor's `2 kHalf` columns of this CTA per row: TMEM at `tcol`,
        // bf16 to `row` (already at the CTA's first column), times `mul`
        auto write_rows = [&](auto cols, uint32_t tcol, uint16_t* row, float mul) {
          constexpr int kHalf = decltype(cols)::value / 2;
          constexpr int N = kHalf < 32 ? kHalf : 32;
#pragma unroll
          for (int c = 0; c < kHalf / N; ++c) {
            uint32_t a[N];
            if (have) {
              tmem_ld_chunk(lane_base + tcol + half * kHalf + c * N, a);
              tmem_ld_wait();
              reg_fence(a);
            } else {
#pragma unroll
              for (int e = 0; e < N; ++e) a[e] = 0u;
            }
#pragma unroll
            for (int q4 = 0; q4 < N / 8; ++q4) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(a[q4 * 8 + 0]) * mul, __uint_as_float(a[q4 * 8 + 1]) * mul);
              v.y = pack_bf16x2(__uint_as_float(a[q4 * 8 + 2]) * mul, __uint_as_float(a[q4 * 8 + 3]) * mul);
              v.z = pack_bf16x2(__uint_as_float(a[q4 * 8 + 4]) * mul, __uint_as_float(a[q4 * 8 + 5]) * mul);
              v.w = pack_bf16x2(__uint_as_float(a[q4 * 8 + 6]) * mul, __uint_as_float(a[q4 * 8 + 7]) * mul);
              if (key < p.n_k)
                *reinterpret_cast<uint4*>(row + half * kHalf + c * N + q4 * 8) = v;
            }
          }
        };
        const long long krow = static_cast<long long>(bh) * p.n_k + key;
        write_rows(std::integral_constant<int, C::kColsV>{}, 256u,
                   p.dv + krow * DV + chunk * C::kColsV, 1.f);
        write_rows(std::integral_constant<int, C::kColsK>{}, C::kDkCol,
                   p.dk + krow * DK + chunk * C::kColsK, p.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace n64

// -D_i = -dO_i . O_i and -lse_i log2(e) (padded rows: 0 and -inf), dQ accumulator = 0.
// kElems values of O and dO per lane (8, or 16 for 512-wide rows), so that a
// row takes at most one warp; each lane also zeroes DK / kLanes of the row's
// fp32 dQ accumulator.
template <int DK, int DV>
__global__ void __launch_bounds__(256) sdpa_bwd_prep(const SdpaBwdPrepParams p) {
  griddep_launch_dependents();   // the main kernel may start its set-up now
  constexpr int kElems = DV > 256 ? DV / 32 : 8;
  constexpr int kLanes = DV / kElems;
  constexpr int kRowsPerBlock = 256 / kLanes;
  constexpr int kZero = DK / kLanes;   // 2 to 16 accumulator floats per lane
  static_assert(kLanes <= 32, "one row per warp at most");
  const int sub = threadIdx.x % kLanes;
  const long long row = static_cast<long long>(blockIdx.x) * kRowsPerBlock + threadIdx.x / kLanes;
  const long long rows = static_cast<long long>(p.b) * p.h * p.n_q_pad;
  if (row >= rows) return;   // whole groups of kLanes lanes leave together
  const long long bh = row / p.n_q_pad;
  const int i = static_cast<int>(row % p.n_q_pad);
  const unsigned group =
      kLanes == 32 ? 0xffffffffu : ((1u << (kLanes % 32)) - 1u) << (threadIdx.x & 31 & ~(kLanes - 1));
  if (i >= p.n_q) {
    if (sub == 0) {
      p.neg_dvec[row] = 0.f;
      p.neg_lse2[row] = -INFINITY;
    }
    return;
  }
  const long long src = (bh * p.n_q + i) * DV + sub * kElems;
  float acc = 0.f;
#pragma unroll
  for (int v8 = 0; v8 < kElems / 8; ++v8) {
    const uint4 o = *reinterpret_cast<const uint4*>(p.out + src + v8 * 8);
    const uint4 g = *reinterpret_cast<const uint4*>(p.dout + src + v8 * 8);
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      acc = fmaf(__uint_as_float(ow[w] << 16), __uint_as_float(gw[w] << 16), acc);
      acc = fmaf(__uint_as_float(ow[w] & 0xffff0000u), __uint_as_float(gw[w] & 0xffff0000u), acc);
    }
  }
  float* z = p.dq_acc + (bh * p.n_q + i) * DK + sub * kZero;
#pragma unroll
  for (int e = 0; e < kZero; e += 2) *reinterpret_cast<float2*>(z + e) = make_float2(0.f, 0.f);
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(group, acc, off);
  if (sub == 0) {
    p.neg_dvec[row] = -acc;
    p.neg_lse2[row] = -p.lse[bh * p.n_q + i] * 1.4426950408889634f;
  }
}

// dQ = scale * accumulator in bf16, 8 elements per thread.
template <int D>
__global__ void __launch_bounds__(256) sdpa_bwd_dq_convert(const SdpaBwdPrepParams p) {
  griddep_wait();   // the main kernel's reduces into the accumulator are complete
  const long long idx = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) * 8;
  const long long n = static_cast<long long>(p.b) * p.h * p.n_q * D;
  if (idx >= n) return;
  const float4 a = *reinterpret_cast<const float4*>(p.dq_acc + idx);
  const float4 c = *reinterpret_cast<const float4*>(p.dq_acc + idx + 4);
  uint4 r;
  r.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
  r.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
  r.z = pack_bf16x2(c.x * p.scale, c.y * p.scale);
  r.w = pack_bf16x2(c.z * p.scale, c.w * p.scale);
  *reinterpret_cast<uint4*>(p.dq + idx) = r;
}

// The prep kernel; reports whether it launched (no query rows: nothing to do).
template <int DK, int DV>
cudaError_t launch_prep(const SdpaBwdPrepParams& pp, cudaStream_t stream, bool* launched) {
  const long long rows = static_cast<long long>(pp.b) * pp.h * pp.n_q_pad;
  *launched = rows > 0;
  if (rows == 0) return cudaSuccess;
  constexpr long long kRowsPerBlock = 256 / (DV / (DV > 256 ? DV / 32 : 8));
  sdpa_bwd_prep<DK, DV><<<static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock), 256, 0,
                          stream>>>(pp);
  return cudaGetLastError();
}

// dQ = scale * accumulator, launched after the main kernel when it ran.
template <int D>
cudaError_t launch_convert(const SdpaBwdPrepParams& pp, cudaStream_t stream, bool after_main) {
  const long long n = static_cast<long long>(pp.b) * pp.h * pp.n_q * D;
  if (n == 0) return cudaSuccess;
  return launch_kernel(sdpa_bwd_dq_convert<D>, dim3(static_cast<unsigned>((n / 8 + 255) / 256)),
                       dim3(256), 0, stream, after_main, pp);
}

template <int DK, int DV>
cudaError_t launch_n64(const SdpaBwdParams& bp, const SdpaBwdPrepParams& pp, cudaStream_t stream) {
  // The main kernel launches with a programmatic dependency on the prep
  // kernel, and the convert kernel on the main one, whenever that kernel was
  // launched: each starts while its predecessor's last CTAs finish and waits
  // (griddep_wait) before reading what it wrote.
  bool prep = false;
  cudaError_t err = launch_prep<DK, DV>(pp, stream, &prep);
  if (err != cudaSuccess) return err;
  const int smem = n64::Cfg<DK, DV>::kSmemBytes;
  err = cudaFuncSetAttribute(n64::sdpa_bwd_tc_n64<DK, DV>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  const long long blocks =
      static_cast<long long>(bp.num_kv_tiles) * bp.b * bp.h * n64::Cfg<DK, DV>::kChunks;
  if (blocks > 0) {
    err = launch_kernel(n64::sdpa_bwd_tc_n64<DK, DV>, dim3(static_cast<unsigned>(blocks)),
                        dim3(n64::kThreads), smem, stream, prep, bp);
    if (err != cudaSuccess) return err;
  }
  return launch_convert<DK>(pp, stream, blocks > 0);
}

// 512-wide heads: the same prep and convert around the kernel of 64-key tiles.
cudaError_t launch_w512(const SdpaBwdParams& bp, const SdpaBwdPrepParams& pp, cudaStream_t stream) {
  bool prep = false;
  cudaError_t err = launch_prep<512, 512>(pp, stream, &prep);
  if (err != cudaSuccess) return err;
  err = launch_sdpa_bwd_w512(bp, prep, stream);
  if (err != cudaSuccess) return err;
  const bool ran = static_cast<long long>(bp.num_kv_tiles) * bp.b * bp.h > 0;
  return launch_convert<512>(pp, stream, ran);
}

}  // namespace

cudaError_t launch_sdpa_bwd(const SdpaBwdParams& bp, const SdpaBwdPrepParams& pp, int d_k, int d_v,
                            cudaStream_t stream) {
  if (d_k == d_v) {
    if (d_k == 16) return launch_n64<16, 16>(bp, pp, stream);
    if (d_k == 32) return launch_n64<32, 32>(bp, pp, stream);
    if (d_k == 64) return launch_n64<64, 64>(bp, pp, stream);
    if (d_k == 128) return launch_n64<128, 128>(bp, pp, stream);
    if (d_k == 256) return launch_n64<256, 256>(bp, pp, stream);
    if (d_k == 512) return launch_w512(bp, pp, stream);
  }
  // Table 3, rows (B): smaller keys than values
  if (d_k == 16 && d_v == 64) return launch_n64<16, 64>(bp, pp, stream);
  if (d_k == 32 && d_v == 64) return launch_n64<32, 64>(bp, pp, stream);
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
