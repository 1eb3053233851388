// Scaled dot-product attention with ONE 128-row query tile per CTA, bf16
// in/out, fp32 accumulation, on the tensor cores.  Same operation and masks
// as the two-tile kernel of sdpa_tc.cu (Eq. (1) of "Attention Is All You
// Need", section 3.2.1, the -infinity mask of section 3.2.3, key padding and
// the restricted window of section 4).  It serves two cases:
//   - wide heads, d_k = d_v in {256, 512} (Table 3, rows (A)), whose 128 x d
//     fp32 O does not fit the two-tile plan in 512 tensor-memory columns:
//       d = 256: key tiles of 64; one CTA per query tile.  All of Q moves
//                into tensor memory, and its 64 KB of shared memory then
//                holds a third stage of K and V.
//       d = 512: key tiles of 64; two CTAs per query tile, one per half of
//                d_v, each recomputing the scores.  Q (128 KB) lands in
//                shared memory; once the softmax warps have copied its
//                first half into tensor memory, that 64 KB holds the
//                second stage of K.  V has one stage.
//   - d = 64 and 128 where the key walk is short: key tiles of 64, 256
//     tensor-memory columns, two CTAs per SM, so short sequences get twice
//     the CTAs in flight and half the serial chain per CTA.  At d = 64 the
//     library may instead pick key tiles of 32 (128 columns, four CTAs per
//     SM) for short walks over many CTAs; the key tile is a template
//     parameter and the K/V boxes must match it.
//   - small heads, d = 16 and 32 on short walks: key tiles of 32, 128
//     tensor-memory columns, four CTAs per SM; rows of 32 or 64 bytes,
//     swizzled at that width.
// Roles:
//   warp 4      TMA producer: Q once, K_j and V_j (this CTA's d_v slice) in
//               two stages each (three at d = 256; at d = 512 K has two and
//               V one).
//   warp 5      MMA issuer (the whole warp; one elected lane issues each
//               instruction): S(j+1) = Q K_{j+1}^T into the free score buffer,
//               then O += P(j) V_j with P(j) read from tensor memory.
//   warps 0-3   softmax, one thread per query row (tensor-memory lane): the
//               running max / sum, P in bf16 over the scores it replaces, the
//               O rescale when the max moves, and the epilogue.
// Tensor memory: score buffers S_0 at 0 and S_1 at BN (fp32, BN keys each),
// O at 2 BN (min(d, 256) fp32 columns).  For d = 256 and 512 the last 128
// columns hold the first 256 columns of Q (bf16 pairs): the softmax warps
// copy their rows there once Q has landed, and those k steps of the scores
// take A from tensor memory.  A score product with A in shared memory
// re-reads the 4 KB of Q per k step and is bound by that read (48 clk at
// N = 64); with A in tensor memory it runs at its compute time (32 clk).
#include "kernels.h"
#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int kBlockM = 128;
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr float kRescaleThreshold = 8.0f;  // log2 units, as in the 64/128 kernel

// KT: keys per tile, 32 or 64 (64 for d >= 128).
template <int DK, int KT>
struct OCfg {
  static constexpr int BN = KT;                             // keys per tile
  static_assert(KT == 32 || (KT == 64 && DK >= 64), "key tile");
  // K has two stages.  At d = 512 (Q alone takes 128 KB) the second lies over
  // the first half of Q, free once the softmax warps have copied it into
  // tensor memory, and V has one stage.
  static constexpr bool kKInQ = DK == 512;
  // At d = 256 all of Q moves to tensor memory, so its 64 KB holds a third
  // stage of K and of V: the loads run two tiles ahead of the products.
  static constexpr bool kKVOverQ = DK == 256;
  static constexpr int kRing = kKVOverQ ? 3 : 2;            // K / V stages (s_full, o_full)
  static constexpr int kKRegionStages = kKInQ ? 1 : 2;     // K stages after Q
  static constexpr int kVStages = kKInQ ? 1 : kRing;
  static_assert(!kKInQ || kRing == 2, "the 512-wide plan indexes its barriers by u & 1");
  static constexpr int kDvc = DK < 256 ? DK : 256;          // O columns per CTA
  static constexpr int kChunks = DK / kDvc;                 // CTAs per query tile
  // Tiles move as boxes of kBoxCols columns, rows of kRowBytes swizzled at
  // that width (128-, 64- or 32-byte swizzle for d >= 64, 32, 16).
  static constexpr int kBoxCols = DK < 64 ? DK : 64;
  static constexpr int kRowBytes = kBoxCols * 2;
  static constexpr uint32_t kLayout = kRowBytes == 128 ? 2u : (kRowBytes == 64 ? 4u : 6u);
  static constexpr uint32_t kSBO = 8 * kRowBytes;           // 8-row group stride
  static constexpr int kStepsPerRow = kRowBytes / 32;       // K=16 steps per swizzled row
  // O columns per TMEM load (16 when four CTAs share an SM at d = 64, to fit 80 registers)
  static constexpr int kOChunk = kDvc < 32 ? kDvc : (DK == 64 && KT == 32 ? 16 : 32);
  static constexpr int kQBox = 128 * kRowBytes;             // kBoxCols columns x 128 rows
  static constexpr int kKVBox = BN * kRowBytes;             // kBoxCols columns x BN rows
  static constexpr int kQBytes = (DK / kBoxCols) * kQBox;
  static constexpr int kKBytes = (DK / kBoxCols) * kKVBox;
  static constexpr int kVBytes = (kDvc / kBoxCols) * kKVBox;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + kKRegionStages * kKBytes;
  static constexpr int kBarOff = kVOff + kVStages * kVBytes;
  // q_full, k_full[kRing], v_full[kRing], s_full[kRing], o_full[kRing],
  // p_full[2], o_last, drain, q_tmem
  static constexpr int kNumBars = 1 + 4 * kRing + 2 + 3;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  static constexpr uint32_t kOCol = 2 * BN;
  static constexpr uint32_t kIdescS = idesc_bf16(kBlockM, BN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(kBlockM, kDvc, false, true);
  static constexpr uint32_t kDescHi = (kSBO >> 4) | (1u << 14) | (kLayout << 29);
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kKOff % 1024 == 0 && kVOff % 1024 == 0 && kKVBox % 1024 == 0, "alignment");
  // d <= 128 fits 256 columns (two CTAs per SM), d <= 32 fits 128 (four)
  static constexpr uint32_t kTmemCols =
      kOCol + kDvc <= 128 ? 128u : (kOCol + kDvc <= 256 ? 256u : 512u);
  static constexpr int kMinBlocks = static_cast<int>(512u / kTmemCols);
  static_assert(kOCol + kDvc <= kTmemCols, "tensor memory");
  // Score k steps whose A operand (Q) sits in tensor memory after O: all of a
  // 256-wide Q, the first half of a 512-wide one (the K half of part 0).
  static constexpr int kQTmemSteps = DK >= 256 ? 16 : 0;
  static constexpr uint32_t kQCol = kOCol + kDvc;
  static_assert(kQCol + kQTmemSteps * 8 <= kTmemCols, "Q in tensor memory");
  // the second K stage fits in the part of Q that tensor memory holds
  static_assert(!kKInQ || kQTmemSteps * 16 / kBoxCols * kQBox >= kKBytes, "K stage over Q");
  static_assert(kQTmemSteps == 0 || (kRowBytes == 128 && (kQTmemSteps * 16) % kBoxCols == 0),
                "Q copied by whole 128-byte-swizzled boxes");
  // the third K and V stage fits in Q, none of which the scores read from shared memory
  static_assert(!kKVOverQ || (kQTmemSteps * 16 == DK && kKBytes + kVBytes <= kQBytes &&
                              kKBytes % 1024 == 0 && !kKInQ),
                "K and V stage over Q");
  static_assert(kSmemBytes * kMinBlocks <= 232448 - 1024 * kMinBlocks, "CTAs per SM");
};

template <int DK, int KT>
__global__ void __launch_bounds__(kThreads, OCfg<DK, KT>::kMinBlocks)
    sdpa_fwd_one_tile(const __grid_constant__ SdpaTcParams p) {
  using C = OCfg<DK, KT>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t smem_base = smem_u32(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bar;
  uint64_t* k_full = bar + 1;
  // A K stage is free again once the scores that read it are done (s_full),
  // a V stage once the O += P V that read it is done (o_full): no separate
  // "empty" barriers, so each key tile costs two commits instead of four.
  // Key tile u uses stage u % kRing and those two barriers of that index; the
  // score buffer and p_full are u & 1.
  constexpr int R = C::kRing;
  uint64_t* v_full = k_full + R;
  uint64_t* s_full = v_full + R;
  uint64_t* o_full = s_full + R;   // o_full[u % R]: one phase per O += P(u) V_u
  uint64_t* p_full = o_full + R;
  uint64_t* o_last = p_full + 2;   // once, after the last O += P V
  uint64_t* drain = o_last + 1;
  uint64_t* q_tmem = drain + 1;    // the softmax warps copied Q into tensor memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_tmem + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const AbortState ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work: units = (batch*head, d_v slice) in groups of p.head_group;
  // inside a group the longest query tiles (causal) go first.  Groups of a
  // few units keep their K and V in L2 on long sequences; when every unit's
  // K and V fit in L2 together the host makes one group of all units, so the
  // longest tiles of the whole grid start first.
  const int units = p.b * p.h * C::kChunks;
  const int nqb = p.num_q_blocks;
  const int head_group = p.head_group;
  const int group_ctas = head_group * nqb;
  const int full_groups = units / head_group;
  const int idx = static_cast<int>(blockIdx.x);
  int g = idx / group_ctas, r = idx % group_ctas, in_group = head_group;
  if (g >= full_groups) {
    g = full_groups;
    r = idx - full_groups * group_ctas;
    in_group = units - full_groups * head_group;
  }
  const int qb = nqb - 1 - r / in_group;
  const int unit = g * head_group + r % in_group;
  const int chunk = unit % C::kChunks;
  const int bh = unit / C::kChunks;
  const int bi = bh / p.h;
  const int hi = bh % p.h;
  const bool causal = (p.mask_kind & 1) != 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < R; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(o_full + s, 1);
      mbar_init(s_full + s, 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(p_full + s, kBlockM);
    mbar_init(o_last, 1);
    mbar_init(drain, 1);
    mbar_init(q_tmem, kBlockM);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, C::kTmemCols);
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
  // Key tile u covers keys [key_base + u BN, key_base + (u + 1) BN), from
  // the first key some row of the tile can see (0 without a restricted
  // window; with one, starting there instead of at a multiple of BN saves
  // the mostly masked tile an aligned grid adds).  Keys past n_k load as
  // zeros and are masked.
  const int qs = qb * kBlockM;
  int key_base = 0, n_kv = 0;
  {
    const int row_hi = min(qs + kBlockM, p.n_q) - 1;
    const int key_lo = max(0, qs - p.win_left);
    int key_hi = min(kv_len, row_hi + 1 + min(p.win_right, p.n_k));
    if (causal) key_hi = min(key_hi, row_hi + 1);
    if (key_hi > key_lo) {
      key_base = key_lo;
      n_kv = (key_hi - key_lo + BN - 1) / BN;
    }
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kv > 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_o);
      mbar_arrive_expect_tx(q_full, C::kQBytes);
      for (int c = 0; c < DK / C::kBoxCols; ++c)
        tma_load_4d(&p.tm_q, q_full, smem + C::kQOff + c * C::kQBox, c * C::kBoxCols, qs, hi, bi);
      int k_issued = 0, v_issued = 0;
      // K stage of tile u (u & 1), and where it lies
      auto k_stage = [&](int u) -> uint8_t* {
        return (u & 1) ? (C::kKInQ ? smem + C::kQOff : smem + C::kKOff + C::kKBytes)
                       : smem + C::kKOff;
      };
      auto load_k = [&](int u) {
        uint8_t* dst = k_stage(u);
        mbar_arrive_expect_tx(k_full + (u & 1), C::kKBytes);
        for (int c = 0; c < DK / C::kBoxCols; ++c)
          tma_load_4d(&p.tm_k, k_full + (u & 1), dst + c * C::kKVBox, c * C::kBoxCols,
                      key_base + u * BN, hi, bi);
      };
      if constexpr (C::kKInQ) {
        // K_{u+1} goes ahead of V_u: it needs only the scores of tile u - 1
        // to be done with its stage, V_u the product of tile u - 1 with V.
        bool go = true;
        load_k(0);
        k_issued = 1;
        for (int u = 0; go && u < n_kv; ++u) {
          const int nk = u + 1;
          if (nk < n_kv) {
            // stage 1's first use: the softmax warps have copied Q's first
            // half into tensor memory; later uses: S(nk - 2) is done
            const bool free_ok = nk == 1 ? mbar_wait(q_tmem, 0, ab)
                                         : mbar_wait(s_full + (nk & 1),
                                                     static_cast<uint32_t>((nk >> 1) - 1) & 1u, ab);
            if (!free_ok) break;
            load_k(nk);
            k_issued = nk + 1;
          }
          // the one V stage: O += P(u-1) V_{u-1} is done with it
          if (u >= 1 && !mbar_wait(o_full + ((u - 1) & 1), static_cast<uint32_t>((u - 1) >> 1) & 1u, ab)) {
            go = false;
            break;
          }
          mbar_arrive_expect_tx(v_full, C::kVBytes);
          for (int c = 0; c < C::kDvc / C::kBoxCols; ++c)
            tma_load_4d(&p.tm_v, v_full, smem + C::kVOff + c * C::kKVBox,
                        chunk * C::kDvc + c * C::kBoxCols, key_base + u * BN, hi, bi);
          v_issued = u + 1;
        }
        mbar_wait_drain(q_full, 0);
        // each load was issued only after the previous one into the same
        // place had been consumed, so only the last of each can be in flight
        for (int u = max(0, k_issued - 2); u < k_issued; ++u)
          mbar_wait_drain(k_full + (u & 1), static_cast<uint32_t>(u >> 1) & 1u);
        if (v_issued > 0) mbar_wait_drain(v_full, static_cast<uint32_t>(v_issued - 1) & 1u);
      } else {
        // K_{u+1} goes ahead of V_u: its stage is free once S(u+1-R) is done,
        // which comes before O += P(u-R) V_{u-R}, the product that frees V_u's.
        auto load_ring_k = [&](int u) -> bool {
          const int s = u % R;
          // S(u-R) read this stage last.  s_full[s] cannot be two phases
          // ahead: S(u) needs the K_u loaded here.
          if (u >= R && !mbar_wait(s_full + s, static_cast<uint32_t>(u / R - 1) & 1u, ab)) return false;
          // the stage over Q: free once the softmax warps have copied Q into
          // tensor memory (the scores never read Q from shared memory here)
          if (C::kKVOverQ && u == 2 && !mbar_wait(q_tmem, 0, ab)) return false;
          uint8_t* kdst = s == 2 ? smem + C::kQOff : smem + C::kKOff + s * C::kKBytes;
          mbar_arrive_expect_tx(k_full + s, C::kKBytes);
          for (int c = 0; c < DK / C::kBoxCols; ++c)
            tma_load_4d(&p.tm_k, k_full + s, kdst + c * C::kKVBox, c * C::kBoxCols, key_base + u * BN,
                        hi, bi);
          k_issued = u + 1;
          return true;
        };
        bool go = load_ring_k(0);
        for (int u = 0; go && u < n_kv; ++u) {
          if (u + 1 < n_kv && !(go = load_ring_k(u + 1))) break;
          const int s = u % R;
          // O += P(u-R) V(u-R) read this stage last; o_full[s] cannot be two
          // phases ahead either (O += P(u) V_u needs V_u).
          if (u >= R && !mbar_wait(o_full + s, static_cast<uint32_t>(u / R - 1) & 1u, ab)) break;
          uint8_t* vdst = s == 2 ? smem + C::kQOff + C::kKBytes : smem + C::kVOff + s * C::kVBytes;
          mbar_arrive_expect_tx(v_full + s, C::kVBytes);
          for (int c = 0; c < C::kDvc / C::kBoxCols; ++c)
            tma_load_4d(&p.tm_v, v_full + s, vdst + c * C::kKVBox, chunk * C::kDvc + c * C::kBoxCols,
                        key_base + u * BN, hi, bi);
          v_issued = u + 1;
        }
        mbar_wait_drain(q_full, 0);
        for (int u = max(0, k_issued - R); u < k_issued; ++u)
          mbar_wait_drain(k_full + u % R, static_cast<uint32_t>(u / R) & 1u);
        for (int u = max(0, v_issued - R); u < v_issued; ++u)
          mbar_wait_drain(v_full + u % R, static_cast<uint32_t>(u / R) & 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop in step (warp-uniform waits and
    // descriptors); one elected lane issues every product and commit.
    if (n_kv > 0) {
      constexpr uint32_t kDescHi = C::kDescHi;
      auto lo = [](uint32_t addr, uint32_t lbo) { return (addr >> 4) | ((lbo >> 4) << 16); };
      const uint32_t q_lo = lo(smem_base + C::kQOff, 16);
      // S(u) = Q K_u^T into score buffer u & 1: waits for K_u in its stage
      // (u & 1; at d = 512 stage 1 lies over the first half of Q), issues the
      // k steps, and commits s_full.
      auto issue_s = [&](int u) -> bool {
        const uint32_t d = tmem + static_cast<uint32_t>((u & 1) * BN);
        const int ks = u % R;
        const uint32_t k_base =
            ks == 0 ? C::kKOff : ((ks == 2 || C::kKInQ) ? C::kQOff : C::kKOff + C::kKBytes);
        const uint32_t b0 = lo(smem_base + k_base, 16);
        if (!mbar_wait_warp(k_full + ks, static_cast<uint32_t>(u / R) & 1u, ab)) return false;
        tc_fence_after();
        constexpr int kSteps = DK / 16;
#pragma unroll
        for (int k = 0; k < kSteps; ++k) {
          constexpr int kS = C::kStepsPerRow;
          const uint32_t bk = b0 + static_cast<uint32_t>(((k / kS) * C::kKVBox + (k % kS) * 32) >> 4);
          if (k < C::kQTmemSteps)
            mma_bf16_ts_warp(d, tmem + C::kQCol + static_cast<uint32_t>(k * 8), bk, kDescHi,
                             C::kIdescS, k > 0 ? 1u : 0u);
          else
            mma_bf16_ss_warp(d, q_lo + static_cast<uint32_t>(((k / kS) * C::kQBox + (k % kS) * 32) >> 4),
                             kDescHi, bk, kDescHi, C::kIdescS, k > 0 ? 1u : 0u);
        }
#ifdef SDPA_TEST_WITHHOLD_FIRST_S_COMMIT
        // (test builds only, never in libsdpa.so: the first score tile is
        // never signalled, so the bounded waits of the softmax warps, and of
        // the producer once it needs that K stage again, run out)
        if (u == 0) return true;
#endif
        mma_commit_warp(s_full + ks);
        return true;
      };
      auto issue_pv = [&](int u) {
        const uint32_t pa = tmem + static_cast<uint32_t>((u & 1) * BN);
        const int stage = C::kVStages == 1 ? 0 : u % R;
        const uint32_t v_base = stage == 2 ? C::kQOff + C::kKBytes : C::kVOff + stage * C::kVBytes;
        const uint32_t b0 = lo(smem_base + v_base, C::kKVBox);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          mma_bf16_ts_warp(tmem + C::kOCol, pa + static_cast<uint32_t>(k * 8),
                           b0 + static_cast<uint32_t>((k * 16 * C::kRowBytes) >> 4), kDescHi,
                           C::kIdescPV,
                           (u > 0 || k > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait_warp(q_full, 0, ab);
      if (C::kQTmemSteps > 0 && ok) ok = mbar_wait_warp(q_tmem, 0, ab);
      tc_fence_after();
      ok = ok && issue_s(0);
      for (int u = 0; ok && u < n_kv; ++u) {
        // S(u+1) into the buffer of P(u-1): PV(u-1) was issued before it.
        const bool next = u + 1 < n_kv;
        if (next && !(ok = issue_s(u + 1))) break;
        const uint32_t vs = C::kVStages == 1 ? 0u : static_cast<uint32_t>(u % R);
        const uint32_t vph = static_cast<uint32_t>(C::kVStages == 1 ? u : u / R) & 1u;
        ok = mbar_wait_warp(p_full + (u & 1), static_cast<uint32_t>(u >> 1) & 1u, ab) &&
             mbar_wait_warp(v_full + vs, vph, ab);
        if (!ok) break;
        tc_fence_after();
        issue_pv(u);
        mma_commit_warp(o_full + u % R);
        if (u + 1 == n_kv) mma_commit_warp(o_last);
      }
      mma_commit_warp(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    const int row = qs + row_in_tile;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float scale_log2 = p.scale_log2;
    const int lo_lim = row - p.win_left;
    const int hi_lim = min(kv_len - 1, causal ? row : row + min(p.win_right, p.n_k));
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    if constexpr (C::kQTmemSteps > 0) {
      // this thread's row of Q, its first kQTmemSteps * 16 columns, into its
      // tensor-memory lane as bf16 pairs (the A layout of a K-major product)
      if (n_kv > 0) {
        ok = mbar_wait_warp(q_full, 0, ab);
        if (ok) {
#pragma unroll 1
          for (int c = 0; c < C::kQTmemSteps * 16 / C::kBoxCols; ++c) {
            const uint8_t* box = smem + C::kQOff + c * C::kQBox;
            uint32_t w[32];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const uint4 v = *reinterpret_cast<const uint4*>(
                  box + sw128_offset(static_cast<uint32_t>(row_in_tile), static_cast<uint32_t>(ch)));
              w[ch * 4 + 0] = v.x;
              w[ch * 4 + 1] = v.y;
              w[ch * 4 + 2] = v.z;
              w[ch * 4 + 3] = v.w;
            }
            tmem_st32(lane_base + C::kQCol + static_cast<uint32_t>(c * 32), w);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(q_tmem);
      }
    }
    for (int u = 0; ok && u < n_kv; ++u) {
      const uint32_t s_col = static_cast<uint32_t>((u & 1) * BN);
      ok = mbar_wait_warp(s_full + u % R, static_cast<uint32_t>(u / R) & 1u, ab);
      if (!ok) break;
      tc_fence_after();
      float s[BN];
      {
        uint32_t sr[32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          tmem_ld32(lane_base + s_col + c * 32, sr);
          tmem_ld_wait();
          reg_fence(sr);
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(sr[e]);
        }
      }
      const int key0 = key_base + u * BN;
      const bool tile_masked = (key0 + BN > kv_len) || (causal && key0 + BN - 1 > qs) ||
                               (key0 + BN - 1 > qs + p.win_right) ||
                               (key0 < qs + kBlockM - 1 - p.win_left);
      if (tile_masked) {
        const int lo_c = lo_lim - key0, hi_c = hi_lim - key0;   // visible columns [lo_c, hi_c]
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c < lo_c || c > hi_c) s[c] = -INFINITY;
      }
      float mx4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx4[i] = s[i];
#pragma unroll
      for (int c = 4; c < BN; c += 8)
#pragma unroll
        for (int i = 0; i < 4; ++i) mx4[i] = fmax3(mx4[i], s[c + i], c + 4 + i < BN ? s[c + 4 + i] : s[c + i]);
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float m_new = fmaxf(m_used, mx * scale_log2);
      float alpha = 1.f;
      bool rescale_warp = false;
      if (u == 0) {
        m_used = m_new;
      } else {
        const bool need = m_new > m_used + kRescaleThreshold;
        rescale_warp = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = ex2_approx(m_used - m_new);
          m_used = m_new;
          l *= alpha;
        }
        // Only a rescale touches O, and it must follow O += P(u-1) V(u-1),
        // whose barrier is o_full[(u-1) % R].  Holding S(u) means
        // O += P(u-2) V(u-2) has landed (S(u) was issued after it), so the
        // barrier's previous phase, u-1-R, is complete; and its next one,
        // u-1+R, is at least O += P(u+1) V(u+1), which needs this softmax's
        // next P.  Its parity wait for the phase of u-1 is therefore exact
        // even though earlier phases were not waited on.
        if (rescale_warp) {
          ok = mbar_wait_warp(o_full + (u - 1) % R, static_cast<uint32_t>((u - 1) / R) & 1u, ab);
          if (!ok) break;
          tc_fence_after();
        }
      }
      const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;
      const float2 sc2 = make_float2(scale_log2, scale_log2);
      const float2 neg2 = make_float2(-m_sub, -m_sub);
      float2 acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
      uint32_t pk[BN / 2];
#pragma unroll
      for (int e = 0; e < BN / 2; ++e) {
        const float2 x = __ffma2_rn(make_float2(s[2 * e], s[2 * e + 1]), sc2, neg2);
        const float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        acc[e & 3] = __fadd2_rn(acc[e & 3], pe);
        pk[e] = pack_bf16x2(pe.x, pe.y);
      }
      if constexpr (BN == 64) {
        tmem_st32(lane_base + s_col, pk);
      } else {
        tmem_st16(lane_base + s_col, pk);
      }
      const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
      if (rescale_warp) {
#pragma unroll
        for (int c = 0; c < C::kDvc / C::kOChunk; ++c) {
          uint32_t o[C::kOChunk];
          tmem_ld_chunk(lane_base + C::kOCol + c * C::kOChunk, o);
          tmem_ld_wait();
          reg_fence(o);
#pragma unroll
          for (int e = 0; e < C::kOChunk; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_chunk(lane_base + C::kOCol + c * C::kOChunk, o);
        }
      }
      l += a.x + a.y;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full + (u & 1));
    }

    // ---- epilogue: O / l -> bf16 -> swizzled staging over Q -> TMA store.
    // Uniform over the warpgroup, so all 128 threads reach the named barrier.
    if (qs < p.n_q) {
      uint8_t* stage = smem + C::kQOff;   // Q is dead once the last product finished
      bool have_o = ok && n_kv > 0;
      if (have_o) {
        have_o = mbar_wait_warp(o_last, 0, ab);
        tc_fence_after();
      }
      if (have_o || (ok && n_kv == 0)) {
        const float inv_l = (have_o && l > 0.f) ? 1.f / l : 0.f;
        if (p.lse != nullptr && chunk == 0 && row < p.n_q)
          p.lse[static_cast<long long>(bh) * p.n_q + row] =
              (have_o && l > 0.f) ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
#pragma unroll
        for (int c = 0; c < C::kDvc / C::kOChunk; ++c) {
          uint32_t o[C::kOChunk];
          if (have_o) {
            tmem_ld_chunk(lane_base + C::kOCol + c * C::kOChunk, o);
            tmem_ld_wait();
            reg_fence(o);
          } else {
#pragma unroll
            for (int e = 0; e < C::kOChunk; ++e) o[e] = 0u;
          }
          const int col0 = c * C::kOChunk;                  // first O column of this chunk
          uint8_t* box = stage + (col0 / C::kBoxCols) * C::kQBox;
#pragma unroll
          for (int q4 = 0; q4 < C::kOChunk / 8; ++q4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l, __uint_as_float(o[q4 * 8 + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l, __uint_as_float(o[q4 * 8 + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l, __uint_as_float(o[q4 * 8 + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l, __uint_as_float(o[q4 * 8 + 7]) * inv_l);
            const uint32_t ch = static_cast<uint32_t>((col0 % C::kBoxCols) / 8 + q4);
            *reinterpret_cast<uint4*>(
                box + swizzle_offset<C::kRowBytes>(static_cast<uint32_t>(row_in_tile), ch)) = v;
          }
        }
        fence_proxy_async_smem();
      }
      named_bar_sync(1, kBlockM);
      if (quarter == 0 && lane == 0 && !*abort_flag) {
        for (int c = 0; c < C::kDvc / C::kBoxCols; ++c)
          tma_store_4d(&p.tm_o, stage + c * C::kQBox, chunk * C::kDvc + c * C::kBoxCols, qs, hi,
                       bi);
        tma_store_commit();
        tma_store_wait_read();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int DK, int KT>
cudaError_t launch_one_tile_impl(const SdpaTcParams& p, cudaStream_t stream) {
  const int smem = OCfg<DK, KT>::kSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(sdpa_fwd_one_tile<DK, KT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  const long long blocks = static_cast<long long>(p.num_q_blocks) * p.b * p.h * OCfg<DK, KT>::kChunks;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  return launch_kernel(sdpa_fwd_one_tile<DK, KT>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads),
                       smem, stream, p.pdl != 0, p);
}

}  // namespace

bool one_tile_supports(int head_dim, int key_tile) {
  switch (head_dim) {
    case 16:
    case 32: return key_tile == 32;
    case 64: return key_tile == 32 || key_tile == 64;
    case 128:
    case 256:
    case 512: return key_tile == 64;
    default: return false;
  }
}

cudaError_t launch_sdpa_one_tile(const SdpaTcParams& p, int head_dim, int key_tile,
                                 cudaStream_t stream) {
  if (!one_tile_supports(head_dim, key_tile)) return cudaErrorInvalidValue;
  switch (head_dim) {
    case 16: return launch_one_tile_impl<16, 32>(p, stream);
    case 32: return launch_one_tile_impl<32, 32>(p, stream);
    case 64: return key_tile == 32 ? launch_one_tile_impl<64, 32>(p, stream)
                                   : launch_one_tile_impl<64, 64>(p, stream);
    case 128: return launch_one_tile_impl<128, 64>(p, stream);
    case 256: return launch_one_tile_impl<256, 64>(p, stream);
    default: return launch_one_tile_impl<512, 64>(p, stream);
  }
}

}  // namespace sdpa
