// Fused scaled dot-product attention, bf16 in/out, fp32 accumulation, on the
// GB300 tensor cores (tcgen05 + TMA + tensor memory): the two-tile kernel.
//
// Operation ("Attention Is All You Need", section 3.2.1, Eq. (1), with the
// decoder's -infinity mask of section 3.2.3, a key-padding mask and the
// restricted window of section 4):
//   O[i, :] = sum_j softmax_j(scale * Q[i, :] . K[j, :]) V[j, :]
// evaluated as an online (streaming) softmax over 128-key tiles, so the
// n_q x n_k score matrix never leaves the SM.  The library runs it for long
// key walks at d = 128 and for keys smaller than values (d_k = 16 or 32 with
// d_v = 64, Table 3 rows (B)); sdpa_one_tile.cu takes the other shapes.
//
// One CTA owns two 128-row query tiles of one (batch, head) and walks the
// key/value tiles once for both:
//   warp 8      TMA producer: Q tiles once, then K_j and V_j into a ring of
//               shared-memory stages (rows swizzled at their width, zero fill
//               past n).
//   warp 9      MMA issuer (the whole warp; one elected lane issues each
//               instruction): S_t = Q_t K_j^T into tensor memory,
//               then O_t += P_t V_j with P_t read from tensor memory, in
//               parts of 64 keys: each starts as soon as the softmax has
//               written that part of P_t.
//   warps 10-11 idle (they complete the third warpgroup for the register split).
//   warps 0-7   two softmax warpgroups, one per query tile, one thread per
//               score row (TMEM lane = row): scale, mask, running max and
//               sum in fp32, exponentials with ex2, P written back to tensor
//               memory as bf16 over the scores it replaces; they also rescale
//               O when the running max grows and run the epilogue.
// The issue order S0(j+1) / PV1(j) / S1(j+1) / PV0(j+1) keeps the tensor core
// busy with one tile while the other tile's softmax runs.
//
// Tensor memory (512 columns): S_0 at 0, S_1 at 128 (fp32, 128 keys each;
// P_t overwrites the first 64 columns of S_t as packed bf16 pairs), O_0 at 256
// and O_1 at 256 + d_v (fp32, d_v columns each).
//
// Running max: the softmax keeps using a stale maximum m_used until a new
// row maximum exceeds it by more than 8 (log2 units), so exp2(x - m_used) <=
// 256 and O needs rescaling only when the maximum really moves.  Both O and
// the running sum use the same m_used, so the final O / l is unchanged.
#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int kBlockM = 128;     // query rows per tile (= tensor-memory lanes)
constexpr int kBlockN = 128;     // keys per tile
constexpr int kThreads = 384;    // 12 warps: two softmax warpgroups + one for TMA/MMA
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// Register split: 384 threads launch with 168 registers each; the TMA/MMA
// warpgroup drops to 64 and the softmax warpgroups rise to 216
// (128 * 64 + 256 * 216 = 63488 <= 384 * 168 = 64512).
constexpr uint32_t kRegsControl = 64;
constexpr uint32_t kRegsSoftmax = 216;
constexpr int kHeadGroup = 8;    // heads whose K/V share L2 at a time
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: a factor of 256
// P_t is handed to the MMA warp in kPParts parts of kBlockN / kPParts keys;
// O_t += P_t V_j starts on a part as soon as the softmax has written it.
constexpr int kPParts = 2;
constexpr int kPPartKeys = kBlockN / kPParts;

// Layout of one operand whose rows hold D bf16 values (Q and K at d_k; V
// and O at d_v).
template <int D>
struct Cfg {
  // Tiles move as boxes of kBoxCols columns x 128 rows, rows of kRowBytes
  // swizzled at that width (128-, 64- or 32-byte swizzle for d >= 64, 32, 16).
  static constexpr int kBoxCols = D < 64 ? D : 64;
  static constexpr int kRowBytes = kBoxCols * 2;
  static constexpr int kBoxBytes = 128 * kRowBytes;
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr uint32_t kLayout = kRowBytes == 128 ? 2u : (kRowBytes == 64 ? 4u : 6u);
  static constexpr uint32_t kSBO = 8 * kRowBytes;          // 8-row group stride
  static constexpr int kStepsPerRow = kRowBytes / 32;      // K=16 steps per swizzled row
  static constexpr int kOChunk = D < 32 ? D : 32;          // O columns per TMEM load
  static constexpr int kTileBytes = kBlockM * D * 2;
  static_assert(D == 16 || D == 32 || D == 64 || D == 128, "head size");
};

// Shared memory of one CTA for key size DK and value size DV: two Q tiles,
// rings of K and V tiles, and the two O tiles' staging for the TMA store
// (over the Q tiles when those are at least as large).
template <int DK, int DV>
struct Plan {
  using CK = Cfg<DK>;
  using CV = Cfg<DV>;
  // K/V ring depths: Q (2 tiles) + K + V stages fill the 227 KB of shared memory.
  static constexpr int kKStages = (DK == 128 || DV == 128) ? 2 : 4;
  static constexpr int kVStages = kKStages;
  static constexpr bool kStageOverQ = CK::kTileBytes >= CV::kTileBytes;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * CK::kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * CK::kTileBytes;
  static constexpr int kVEnd = kVOff + kVStages * CV::kTileBytes;
  static constexpr int kStageOff = kStageOverQ ? kQOff : kVEnd;
  static constexpr int kBarOff = kStageOverQ ? kVEnd : kVEnd + 2 * CV::kTileBytes;
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 6 + 2 * (kPParts - 1) + 1;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  static constexpr uint32_t kIdescS = idesc_bf16(kBlockM, kBlockN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(kBlockM, DV, false, true);
  static_assert(kSmemBytes <= 232448, "shared memory");
};

struct Bars {
  uint64_t* q_full;
  uint64_t* k_full;
  uint64_t* k_empty;
  uint64_t* v_full;
  uint64_t* v_empty;
  uint64_t* s_full;   // [2]
  uint64_t* p_part;   // [2 * (kPParts - 1)]: parts of P_t written (the last part signals p_full)
  uint64_t* p_full;   // [2]
  uint64_t* o_full;   // [2]
  uint64_t* drain;
};

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
sdpa_fwd_bf16_tc(const __grid_constant__ SdpaTcParams p) {
  using C = Plan<DK, DV>;
  using CK = Cfg<DK>;
  using CV = Cfg<DV>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms.
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t smem_base = smem_u32(smem);

  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  Bars bars;
  bars.q_full = bar_mem;
  bars.k_full = bar_mem + 1;
  bars.k_empty = bars.k_full + C::kKStages;
  bars.v_full = bars.k_empty + C::kKStages;
  bars.v_empty = bars.v_full + C::kVStages;
  bars.s_full = bars.v_empty + C::kVStages;
  bars.p_part = bars.s_full + 2;
  bars.p_full = bars.p_part + 2 * (kPParts - 1);
  bars.o_full = bars.p_full + 2;
  bars.drain = bars.o_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars.drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const AbortState ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work assignment.  CTAs take heads in groups of kHeadGroup so that the
  // K/V of the heads in flight stay in L2; inside a group the longest query
  // blocks (causal) go first.
  const int bh_count = p.b * p.h;
  const int nqb = p.num_q_blocks;
  const int group_ctas = kHeadGroup * nqb;
  const int full_groups = bh_count / kHeadGroup;
  const int idx = static_cast<int>(blockIdx.x);
  int g = idx / group_ctas, r = idx % group_ctas, heads_in_group = kHeadGroup;
  if (g >= full_groups) {
    g = full_groups;
    r = idx - full_groups * group_ctas;
    heads_in_group = bh_count - full_groups * kHeadGroup;
  }
  const int qb = nqb - 1 - r / heads_in_group;
  const int bh = g * kHeadGroup + r % heads_in_group;
  const int bi = bh / p.h;
  const int hi = bh % p.h;
  const bool causal = (p.mask_kind & 1) != 0;

  // ---- set-up: barriers (one thread), tensor memory (MMA warp)
  if (threadIdx.x == 0) {
    mbar_init(bars.q_full, 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bars.k_full + s, 1);
      mbar_init(bars.k_empty + s, 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bars.v_full + s, 1);
      mbar_init(bars.v_empty + s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.s_full + t, 1);
      for (int q = 0; q + 1 < kPParts; ++q) mbar_init(bars.p_part + t * (kPParts - 1) + q, kBlockM);
      mbar_init(bars.p_full + t, kBlockM);
      mbar_init(bars.o_full + t, 1);
    }
    mbar_init(bars.drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every CTA holds its tensor memory now: the next kernel in the stream may
  // launch; this grid's inputs may come from the previous one, so wait for it.
  griddep_launch_dependents();
  griddep_wait();
  // The key-padding lengths may come from the previous kernel in the
  // stream: read them only after griddep_wait().
  int kv_len = p.n_k;
  if ((p.mask_kind & 2) && p.kv_lengths != nullptr) {
    kv_len = p.kv_lengths[bi];
    kv_len = kv_len < 0 ? 0 : (kv_len > p.n_k ? p.n_k : kv_len);
  }
  // Query tile t covers rows [q0 + 128 t, q0 + 128 t + 128).  It needs the key
  // tiles [lo_of(t), hi_of(t)): those holding at least one key that some
  // row of the tile can see (causal, padding and restricted-window limits).
  const int q0 = qb * 2 * kBlockM;
  auto tile_range = [&](int t) -> int2 {
    const int qs = q0 + t * kBlockM;
    if (qs >= p.n_q) return make_int2(0, 0);
    const int row_hi = min(qs + kBlockM, p.n_q) - 1;
    int key_lo = max(0, qs - p.win_left);
    int key_hi = min(kv_len, row_hi + 1 + min(p.win_right, p.n_k));
    if (causal) key_hi = min(key_hi, row_hi + 1);
    if (key_hi <= key_lo) return make_int2(0, 0);
    return make_int2(key_lo / kBlockN, (key_hi + kBlockN - 1) / kBlockN);
  };
  const int2 range0 = tile_range(0), range1 = tile_range(1);
  auto lo_of = [&](int t) { return t ? range1.x : range0.x; };
  auto hi_of = [&](int t) { return t ? range1.y : range0.y; };
  const bool has0 = range0.y > range0.x, has1 = range1.y > range1.x;
  // the CTA walks key tiles [j_first, j_first + n_kv)
  const int j_first = has0 ? (has1 ? min(range0.x, range1.x) : range0.x) : (has1 ? range1.x : 0);
  const int j_end = has0 ? (has1 ? max(range0.y, range1.y) : range0.y) : (has1 ? range1.y : 0);
  const int n_kv = j_end - j_first;
  auto active = [&](int t, int j) { return j >= lo_of(t) && j < hi_of(t); };

  if (warp >= 8) {
   regs_decrease<kRegsControl>();
   if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_o);
      uint32_t q_bytes = 0;
      q_bytes += has0 ? CK::kTileBytes : 0;
      q_bytes += has1 ? CK::kTileBytes : 0;
      if (q_bytes > 0) {
        mbar_arrive_expect_tx(bars.q_full, q_bytes);
        for (int t = 0; t < 2; ++t) {
          if (hi_of(t) <= lo_of(t)) continue;
          for (int c = 0; c < CK::kBoxes; ++c)
            tma_load_4d(&p.tm_q, bars.q_full, smem + C::kQOff + t * CK::kTileBytes + c * CK::kBoxBytes,
                        c * CK::kBoxCols, q0 + t * kBlockM, hi, bi);
        }
      }
      int k_issued = 0, v_issued = 0;  // tiles whose K (V) copy was started
      for (int u = 0; u < n_kv; ++u) {
        const int j = j_first + u;
        const int sk = u % C::kKStages;
        const uint32_t uk = static_cast<uint32_t>(u / C::kKStages);
        if (u >= C::kKStages && !mbar_wait(bars.k_empty + sk, (uk - 1) & 1u, ab)) break;
        mbar_arrive_expect_tx(bars.k_full + sk, CK::kTileBytes);
        for (int c = 0; c < CK::kBoxes; ++c)
          tma_load_4d(&p.tm_k, bars.k_full + sk,
                      smem + C::kKOff + sk * CK::kTileBytes + c * CK::kBoxBytes, c * CK::kBoxCols,
                      j * kBlockN, hi, bi);
        k_issued = u + 1;
        const int sv = u % C::kVStages;
        const uint32_t uv = static_cast<uint32_t>(u / C::kVStages);
        if (u >= C::kVStages && !mbar_wait(bars.v_empty + sv, (uv - 1) & 1u, ab)) break;
        mbar_arrive_expect_tx(bars.v_full + sv, CV::kTileBytes);
        for (int c = 0; c < CV::kBoxes; ++c)
          tma_load_4d(&p.tm_v, bars.v_full + sv,
                      smem + C::kVOff + sv * CV::kTileBytes + c * CV::kBoxBytes, c * CV::kBoxCols,
                      j * kBlockN, hi, bi);
        v_issued = u + 1;
      }
      // Let every copy this thread started land before the CTA can exit.
      if (q_bytes > 0) mbar_wait_drain(bars.q_full, 0);
      for (int j = max(0, k_issued - C::kKStages); j < k_issued; ++j)
        mbar_wait_drain(bars.k_full + j % C::kKStages, static_cast<uint32_t>(j / C::kKStages) & 1u);
      for (int j = max(0, v_issued - C::kVStages); j < v_issued; ++j)
        mbar_wait_drain(bars.v_full + j % C::kVStages, static_cast<uint32_t>(j / C::kVStages) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop in step (warp-uniform waits and
    // descriptors); one elected lane issues every product and commit.
    if (n_kv > 0) {
      const uint32_t q_smem = smem_base + C::kQOff;
      const uint32_t k_smem = smem_base + C::kKOff;
      const uint32_t v_smem = smem_base + C::kVOff;
      // Descriptors split in halves: the high word is fixed by the layout, the
      // low word holds (address >> 4) and the leading offset; a K step adds
      // its byte offset >> 4 to the low word (no carry: smem < 256 KB).
      const uint64_t kq = smem_desc(q_smem, 16, CK::kSBO, CK::kLayout);
      const uint64_t kk = smem_desc(k_smem, 16, CK::kSBO, CK::kLayout);
      const uint64_t kv = smem_desc(v_smem, CV::kBoxBytes, CV::kSBO, CV::kLayout);
      const uint32_t q_lo = static_cast<uint32_t>(kq), qk_hi = static_cast<uint32_t>(kq >> 32);
      const uint32_t k_lo = static_cast<uint32_t>(kk);
      const uint32_t v_lo = static_cast<uint32_t>(kv), v_hi = static_cast<uint32_t>(kv >> 32);
      auto issue_s = [&](int t, int stage) {
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(t * kBlockN);
        const uint32_t a0 = q_lo + static_cast<uint32_t>((t * CK::kTileBytes) >> 4);
        const uint32_t b0 = k_lo + static_cast<uint32_t>((stage * CK::kTileBytes) >> 4);
#pragma unroll
        for (int k = 0; k < DK / 16; ++k) {
          const uint32_t off = static_cast<uint32_t>(
              ((k / CK::kStepsPerRow) * CK::kBoxBytes + (k % CK::kStepsPerRow) * 32) >> 4);
          mma_bf16_ss_warp(d_tmem, a0 + off, qk_hi, b0 + off, qk_hi, C::kIdescS, k > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t V_j over keys [16 k_begin, 16 k_end) of the tile.
      auto issue_pv = [&](int t, int stage, bool accumulate, int k_begin, int k_end) {
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(256 + t * DV);
        const uint32_t p_tmem = tmem + static_cast<uint32_t>(t * kBlockN);
        const uint32_t b0 = v_lo + static_cast<uint32_t>((stage * CV::kTileBytes) >> 4);
#pragma unroll
        for (int k = k_begin; k < k_end; ++k) {
          mma_bf16_ts_warp(d_tmem, p_tmem + static_cast<uint32_t>(k * 8),
                           b0 + static_cast<uint32_t>((k * 16 * CV::kRowBytes) >> 4), v_hi, C::kIdescPV,
                           (accumulate || k > 0) ? 1u : 0u);
        }
      };

      bool ok = mbar_wait_warp(bars.q_full, 0, ab) && mbar_wait_warp(bars.k_full, 0, ab);
      tc_fence_after();
      if (ok) {
        const int last_t = active(1, j_first) ? 1 : 0;
        for (int t = 0; t < 2; ++t) {
          if (!active(t, j_first)) continue;
          issue_s(t, 0);
#ifdef SDPA_TEST_WITHHOLD_FIRST_S_COMMIT
          // Test builds only (never in libsdpa.so): the first score tile of
          // query tile 0 is never signalled, so its softmax warps' bounded
          // wait runs out and the kernel reports a timeout.
          if (t != 0) mma_commit_warp(bars.s_full + t);
#else
          mma_commit_warp(bars.s_full + t);
#endif
          if (t == last_t) mma_commit_warp(bars.k_empty);
        }
      }
      for (int u = 0; ok && u < n_kv; ++u) {
        const int j = j_first + u;
        const int s = u % C::kVStages;
        ok = mbar_wait_warp(bars.v_full + s, static_cast<uint32_t>(u / C::kVStages) & 1u, ab);
        if (!ok) break;
        tc_fence_after();
        const bool pv_any = active(0, j) || active(1, j);
        const bool s_any = active(0, j + 1) || active(1, j + 1);
        const int last_pv_t = active(1, j) ? 1 : 0;
        const int last_s_t = active(1, j + 1) ? 1 : 0;
        const int sn = (u + 1) % C::kKStages;
        const uint32_t kn_phase = static_cast<uint32_t>((u + 1) / C::kKStages) & 1u;
        bool k_next_ready = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if (active(t, j)) {
            // P_t V_j starts on the first parts of P_t while the softmax
            // still computes the later ones.
            const uint32_t pp = static_cast<uint32_t>(j - lo_of(t)) & 1u;
            constexpr int kSteps = kPPartKeys / 16;
#pragma unroll
            for (int q = 0; q < kPParts && ok; ++q) {
              ok = mbar_wait_warp(q + 1 < kPParts ? bars.p_part + t * (kPParts - 1) + q : bars.p_full + t, pp, ab);
              if (!ok) break;
              tc_fence_after();
              issue_pv(t, s, q > 0 || j > lo_of(t), q * kSteps, (q + 1) * kSteps);
            }
            if (!ok) break;
            mma_commit_warp(bars.o_full + t);
            if (t == last_pv_t) mma_commit_warp(bars.v_empty + s);
          }
          if (active(t, j + 1)) {
            if (!k_next_ready) {
              ok = mbar_wait_warp(bars.k_full + sn, kn_phase, ab);
              if (!ok) break;
              tc_fence_after();
              k_next_ready = true;
            }
            issue_s(t, sn);
            mma_commit_warp(bars.s_full + t);
            if (t == last_s_t) mma_commit_warp(bars.k_empty + sn);
          }
        }
        // A key tile inside the walked range that no query tile uses is still
        // released, so the producer's ring keeps turning.
        if (ok && !pv_any) mma_commit_warp(bars.v_empty + s);
        if (ok && !s_any && u + 1 < n_kv) {
          ok = mbar_wait_warp(bars.k_full + sn, kn_phase, ab);
          if (ok) mma_commit_warp(bars.k_empty + sn);
        }
      }
      // Every MMA issued above has finished once this barrier completes.
      mma_commit_warp(bars.drain);
      mbar_wait_drain(bars.drain, 0);
    }
   }
  } else {
    regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;           // query tile of this warpgroup
    const int quarter = warp & 3;      // TMEM lane quarter of this warp
    const int row_in_tile = quarter * 32 + lane;
    const int q_start_t = q0 + t * kBlockM;
    const int row = q_start_t + row_in_tile;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = static_cast<uint32_t>(t * kBlockN);
    const uint32_t o_col = static_cast<uint32_t>(256 + t * DV);
    const float scale_log2 = p.scale_log2;
    const int t_lo = lo_of(t), t_hi = hi_of(t);
    const int n_t = t_hi - t_lo;
    // visible keys of this row: [lo_lim, hi_lim]
    const int lo_lim = row - p.win_left;
    const int hi_lim = min(kv_len - 1, causal ? row : row + min(p.win_right, p.n_k));

    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = t_lo; j < t_hi; ++j) {
      const uint32_t it = static_cast<uint32_t>(j - t_lo);   // this tile's iteration
      ok = mbar_wait_warp(bars.s_full + t, it & 1u, ab);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + s_col + c * 32, sr[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence(sr[c]);
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);

      const int key0 = j * kBlockN;
      const bool tile_masked = (key0 + kBlockN > kv_len) ||
                               (causal && key0 + kBlockN - 1 > q_start_t) ||
                               (key0 + kBlockN - 1 > q_start_t + p.win_right) ||
                               (key0 < q_start_t + kBlockM - 1 - p.win_left);
      if (tile_masked) {
        const int lo = lo_lim - key0, hi_c = hi_lim - key0;  // visible columns [lo, hi_c]
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < lo || c > hi_c) s[c] = -INFINITY;
      }
      // Row maximum: eight independent chains of three-input max.
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = fmax3(s[i], s[8 + i], s[16 + i]);
#pragma unroll
      for (int c = 24; c + 16 <= 120; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + 8 + i]);
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[120 + i]);
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7]));
      const float m_new = fmaxf(m_used, mx * scale_log2);
      // Move the reference maximum only when it grew by more than the
      // threshold (always on the first tile, where O holds nothing yet).
      float alpha = 1.f;
      bool rescale_warp = false;
      if (it == 0) {
        m_used = m_new;
      } else {
        const bool need = m_new > m_used + kRescaleThreshold;
        rescale_warp = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = ex2_approx(m_used - m_new);
          m_used = m_new;
          l *= alpha;
        }
      }
      // O_t already holds P(j-1) V(j-1): the commit that signalled S_t(j)
      // covers every MMA issued before it, PV_t(j-1) included.  The rescale
      // comes before the first half of P is released, since P(j) V(j) then
      // starts to accumulate into O_t.
      // (16-column chunks: the 128 scores are live here.)
      if (rescale_warp) {
#pragma unroll
        for (int c = 0; c < DV / 16; ++c) {
          uint32_t o[16];
          tmem_ld_chunk(lane_base + o_col + c * 16, o);
          tmem_ld_wait();
          reg_fence(o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_chunk(lane_base + o_col + c * 16, o);
        }
      }
      const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;
      // p = exp2(s * scale * log2(e) - m): one packed FMA per pair of scores,
      // four independent packed partial sums.
      const float2 sc2 = make_float2(scale_log2, scale_log2);
      const float2 neg2 = make_float2(-m_sub, -m_sub);
      float2 acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kPParts; ++q) {
        uint32_t pk[kPPartKeys / 2];
#pragma unroll
        for (int e = 0; e < kPPartKeys / 2; ++e) {
          const int c = q * kPPartKeys + 2 * e;
          const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sc2, neg2);
          const float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          acc[e & 3] = __fadd2_rn(acc[e & 3], pe);
          pk[e] = pack_bf16x2(pe.x, pe.y);
        }
        tmem_st_chunk(lane_base + s_col + q * (kPPartKeys / 2), pk);
        if (q + 1 < kPParts) {
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bars.p_part + t * (kPParts - 1) + q);
        }
      }
      const float2 a01 = __fadd2_rn(acc[0], acc[1]);
      const float2 a23 = __fadd2_rn(acc[2], acc[3]);
      const float2 a = __fadd2_rn(a01, a23);
      const float rowsum = a.x + a.y;
      l += rowsum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bars.p_full + t);
    }

    // ---- epilogue: O / l -> bf16 -> swizzled staging (over Q_t when it is at
    // least as large, else a region of its own) -> TMA store.
    // The branch is uniform over the warpgroup, so all 128 threads reach the
    // named barrier; a warp whose waits failed skips only its own writes.
    if (q_start_t < p.n_q) {
      uint8_t* stage = smem + C::kStageOff + t * CV::kTileBytes;
      bool have_o = ok && n_t > 0;
      if (have_o) {
        have_o = mbar_wait_warp(bars.o_full + t, static_cast<uint32_t>(n_t - 1) & 1u, ab);
        tc_fence_after();
      }
      if (have_o || (ok && n_t == 0)) {
        const float inv_l = (have_o && l > 0.f) ? 1.f / l : 0.f;
        if (p.lse != nullptr && row < p.n_q) {
          // natural log-sum-exp of the row's scaled scores (for the backward)
          p.lse[static_cast<long long>(bh) * p.n_q + row] =
              (have_o && l > 0.f) ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
#pragma unroll
        for (int c = 0; c < DV / CV::kOChunk; ++c) {
          uint32_t o[CV::kOChunk];
          if (have_o) {
            tmem_ld_chunk(lane_base + o_col + c * CV::kOChunk, o);
            tmem_ld_wait();
            reg_fence(o);
          } else {
#pragma unroll
            for (int e = 0; e < CV::kOChunk; ++e) o[e] = 0u;
          }
          const int col0 = c * CV::kOChunk;                // first O column of this chunk
          uint8_t* box = stage + (col0 / CV::kBoxCols) * CV::kBoxBytes;
#pragma unroll
          for (int q4 = 0; q4 < CV::kOChunk / 8; ++q4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l, __uint_as_float(o[q4 * 8 + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l, __uint_as_float(o[q4 * 8 + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l, __uint_as_float(o[q4 * 8 + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l, __uint_as_float(o[q4 * 8 + 7]) * inv_l);
            const uint32_t chunk = static_cast<uint32_t>((col0 % CV::kBoxCols) / 8 + q4);
            *reinterpret_cast<uint4*>(
                box + swizzle_offset<CV::kRowBytes>(static_cast<uint32_t>(row_in_tile), chunk)) = v;
          }
        }
        fence_proxy_async_smem();
      }
      named_bar_sync(1 + t, 128);
      if (quarter == 0 && lane == 0 && !*abort_flag) {
        for (int c = 0; c < CV::kBoxes; ++c)
          tma_store_4d(&p.tm_o, stage + c * CV::kBoxBytes, c * CV::kBoxCols, q_start_t, hi, bi);
        tma_store_commit();
        tma_store_wait_read();
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int DK, int DV>
cudaError_t launch_impl(const SdpaTcParams& p, cudaStream_t stream) {
  const int smem = Plan<DK, DV>::kSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(sdpa_fwd_bf16_tc<DK, DV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  const long long blocks = static_cast<long long>(p.num_q_blocks) * p.b * p.h;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  return launch_kernel(sdpa_fwd_bf16_tc<DK, DV>, dim3(static_cast<unsigned>(blocks)),
                       dim3(kThreads), smem, stream, p.pdl != 0, p);
}

}  // namespace

cudaError_t launch_sdpa_tc(const SdpaTcParams& p, int d_k, int d_v, cudaStream_t stream) {
  if (d_k == d_v) {
    if (d_k == 16) return launch_impl<16, 16>(p, stream);
    if (d_k == 32) return launch_impl<32, 32>(p, stream);
    if (d_k == 64) return launch_impl<64, 64>(p, stream);
    if (d_k == 128) return launch_impl<128, 128>(p, stream);
  }
  // Table 3, rows (B): smaller keys than values
  if (d_k == 16 && d_v == 64) return launch_impl<16, 64>(p, stream);
  if (d_k == 32 && d_v == 64) return launch_impl<32, 64>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
