// prefill_pair.cu -- exact attention forward (FMHA) on CTA pairs: one tcgen05
// MMA of M = 256 serves the query tiles of two CTAs.  Used for head dim 256
// (head dim 128 runs faster on single CTAs with two query tiles, prefill.cu).
//
// A cluster of two CTAs takes 256 query rows of one (batch, query head); CTA r
// holds rows [128r, 128r + 128) of them.  Rank 0's MMA warp issues every
// MMA for the pair (cta_group::2):
//   S = Q K^T    A = Q from each CTA's shared memory (its 128 rows), B = the
//                128-key K tile, split by keys: CTA r holds keys [64r, 64r+64);
//   O += P V     A = P from each CTA's TMEM (its 128 rows), B = the V tile,
//                split by head-dim columns: CTA r holds columns [r*d/2, (r+1)*d/2).
// Each CTA receives its 128 rows of S and O in its own TMEM.  Compared with one
// CTA computing two query tiles, every SM reads half the K and V bytes from L2,
// issues half the MMA instructions per key, and re-reads its Q operand from
// shared memory half as often per FLOP (the B half of each MMA is half as wide),
// and the freed TMEM holds two (d = 256) or three (d = 128) S buffers, so the
// MMA warp runs one or two KV tiles ahead of the softmax.  Signals between the
// two SMs of a pair are slow under load (a multicast commit or a remote arrive
// took about 2000 cycles to be seen while the pair's MMAs were running), so
// the deeper the S buffering the better those latencies are hidden.
//
// Warp roles in each CTA (4 NWG + 4 warps):
//   * softmax warps, NWG warpgroups on the CTA's 128 rows (thread = row; NWG = 4
//       for d = 128, 2 for d = 256): warpgroup h takes the key columns
//       [h 128/NWG, (h+1) 128/NWG) of every S tile; the warpgroups exchange
//       their partial row maxima through shared memory, keep the running max m
//       and their partial row sums, rescale their share of the O columns in
//       TMEM when m grows by more than 2^8, write P (bf16) over their S
//       columns, and finally normalise and store their share of O (and LSE);
//   * the next warp: TMEM allocation for the pair; in rank 0 also the MMA issuer;
//   * the next: TMA producer: this CTA's Q tile once, then its K and V halves
//       of every KV tile, into rings of 2 (d = 256) or 3 (d = 128) stages.
//       Every copy's bytes complete on rank 0's barrier, so rank 0's MMA warp
//       starts a tile only when both halves are in place.
//   * two more warps idle (the control warps form one warpgroup).
// Completion of each MMA group is multicast to the barriers of both CTAs; the
// softmax warps of rank 1 publish P to rank 0's barrier with remote arrivals.
//
// The algorithm is the online softmax of "60 . r57 -- FA KV staging double
// buffering (REVERTED)", section 2.3, on the kernel shape of "STAGE_D.md --
// FMHA Kernel Development", Architecture, TMEM Layout and P Staging Paths (P
// kept in TMEM as the A operand of the P.V MMA); the in-kernel normalisation,
// natural-log LSE and the rescale threshold are those of prefill.cu.
//
// TMEM columns per CTA (512 allocated for the pair): O at [0, d), S buffer b
// at d + 128 b.  P of warpgroup h's keys of a tile occupies the first half of
// that warpgroup's own S columns (bf16 pairs).  Issue order per KV tile j:  S(j + NS - 1), then P(j).V(j).  With
// three S buffers the softmax of tile j may find P(j-2).V(j-2) still running,
// so P.V(j) completes on O barrier j % 2: the rescale's wait for P(j-1).V(j-1)
// is then never more than one phase ahead of its barrier.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when m grows by > 2^8

template <int D>
struct PairCfg {
  static constexpr int BN = kPrefillKVStageRows;           // keys per KV tile (= S columns)
  static constexpr int NS = (D == 128) ? 3 : 2;            // S buffers
  static constexpr int kLook = NS - 1;                     // KV tiles the S MMAs run ahead
  static constexpr int kPanels = D / 64;                   // 128-byte panels per row of Q / K
  static constexpr int kQPanelBytes = kPrefillTileM * 128;
  static constexpr int kQBytes = kPanels * kQPanelBytes;   // this CTA's Q tile
  static constexpr int kKRows = BN / 2;                    // K rows of a tile held by one CTA
  static constexpr int kKPanelBytes = kKRows * 128;
  static constexpr int kKStageBytes = kPanels * kKPanelBytes;
  static constexpr int kVPanels = D / 128;                 // V panels (64 columns) held by one CTA
  static constexpr int kVPanelBytes = BN * 128;
  static constexpr int kVStageBytes = kVPanels * kVPanelBytes;
  // softmax warpgroups per CTA: two 64-column slices (four 32-column slices were
  // measured no faster at d = 128, and at d = 256 the larger O share of a
  // warpgroup does not fit the four-warpgroup register budget)
  static constexpr int NWG = 2;
  static constexpr int kCols = BN / NWG;                   // S columns (keys) per warpgroup
  static_assert(kCols == 32 || kCols == 64, "one or two 32-column TMEM loads per tile");
  static constexpr int kStagesK = (D == 128) ? 3 : 2;
  static constexpr int kStagesV = (D == 128) ? 3 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + kStagesK * kKStageBytes;
  static constexpr int kRedOff = kVOff + kStagesV * kVStageBytes;
  // row-max exchange [2 tiles in flight][NWG warpgroups][128 rows] and the final
  // row sums [2 sums][NWG warpgroups][128 rows], fp32
  static constexpr int kRedBytes = 2 * 2 * NWG * 128 * 4;
  static constexpr int kBarOff = kRedOff + kRedBytes;
  // barriers: fullQ, fullK[SK], emptyK[SK], fullV[SV], emptyV[SV], S[NS], P[NS], O[2], Fin
  static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + 2 * NS + 3;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  static constexpr int kSoftWarps = 4 * NWG;
  static constexpr int kThreads = (kSoftWarps + 4) * 32;
  static constexpr int kMmaWarp = kSoftWarps;
  static constexpr int kTmaWarp = kSoftWarps + 1;
  // With two softmax warpgroups, 12 warps launch with 168 registers each: the
  // control warpgroup drops to 80, the softmax warpgroups grow to 208
  // (8*32*208 + 4*32*80 = 63488 <= 64512).  With four, the launch's ~100
  // registers per thread suffice for 32 columns and no split is made.
  static constexpr int kSoftmaxRegs = 208;
  static constexpr int kCtlRegs = 80;
  static_assert(NWG != 2 || (8 * kSoftmaxRegs + 4 * kCtlRegs) * 32 <= kThreads * 168, "register split");
  static constexpr uint32_t kTmemCols = 512;
  __host__ __device__ static constexpr uint32_t o_col() { return 0u; }
  __host__ __device__ static constexpr uint32_t s_col(int buf) { return (uint32_t)(D + buf * BN); }
  static_assert(D + NS * BN <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  // softmax arrivals on a P barrier: every softmax warp of both CTAs
  static constexpr uint32_t kPArrivals = 2 * kSoftWarps;
};

template <int NTHREADS>
__device__ __forceinline__ void softmax_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NTHREADS) : "memory");  // the softmax warps of this CTA
}

// WIN: causal sliding window with attention sinks (window, n_sink); without it
// both are ignored and the tile list is every KV tile
template <int D, bool WIN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<D>::kThreads, 1)
    fmha_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o_ptr,
                     float* __restrict__ lse_ptr, int Hq, int Hkv, int Sq_max, int Skv_max, int causal,
                     int o_bf16, float scale, int n_units_per_head_batch, uint32_t* err,
                     const int* __restrict__ cu_q, const int* __restrict__ kv_lens, int total_q,
                     int window, int n_sink) {
  using C = PairCfg<D>;
  constexpr int BN = C::BN, NS = C::NS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  // ---- work unit of the pair: longest causal work first ----
  const int HB = n_units_per_head_batch;  // Hq * B
  const int n_blocks_q = (Sq_max + 2 * kPrefillTileM - 1) / (2 * kPrefillTileM);
  const int pair = blockIdx.x >> 1;
  // causal: heaviest query blocks first; non-causal: the query blocks of one head
  // are neighbours, so that head's K/V stay in L2 while they run
  const int qb = causal ? (n_blocks_q - 1 - pair / HB) : (pair % n_blocks_q);
  const int hb = causal ? pair % HB : pair / n_blocks_q;
  const int hq = hb % Hq, b = hb / Hq;
  const int hk = hq / (Hq / Hkv);
  // this sequence's query rows and keys (fixed-length or packed varlen batch)
  const SeqExtent ext = seq_extent(b, Sq_max, Skv_max, cu_q, kv_lens, total_q);
  const int Sq = ext.Sq, Skv = ext.Skv;
  const int q0_pair = qb * 2 * kPrefillTileM;
  const int q0 = q0_pair + (int)rank * kPrefillTileM;  // this CTA's first query row
  const long long off = (long long)Skv - Sq;            // bottom-right causal alignment
  // KV tiles of the pair (both CTAs compute the same count)
  int n_kv;
  {
    int kv_hi = Skv;
    if (causal) {
      const long long q_last = (long long)min(Sq, q0_pair + 2 * kPrefillTileM) - 1;
      const long long hi = q_last + off + 1;
      kv_hi = (int)(hi < 0 ? 0 : (hi > Skv ? Skv : hi));
    }
    n_kv = (kv_hi + BN - 1) / BN;
    if (q0_pair >= Sq) n_kv = 0;  // a q-block past the end of this sequence (varlen)
  }
  // with a sliding window the loops run over a list of KV tiles (list index j, key
  // tile tile_list_key(tl, j)); both CTAs of the pair derive the same list
  const TileList tl = WIN ? tile_list((long long)q0_pair + off, n_kv, window, n_sink, Skv, BN)
                          : TileList{0x7FFFFFFF, 0};
  n_kv = tile_list_len(tl, n_kv);
  // every existing row of this CTA admits keys [0, kv_lo): tiles past it need a mask
  int kv_lo = Skv;
  if (causal) {
    const long long lo = (long long)q0 + off + 1;
    kv_lo = (int)(lo < 0 ? 0 : (lo > Skv ? Skv : lo));
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  float* red = reinterpret_cast<float*>(smem + C::kRedOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_q = bars;
  uint64_t* bar_fullK = bars + 1;
  uint64_t* bar_emptyK = bar_fullK + C::kStagesK;
  uint64_t* bar_fullV = bar_emptyK + C::kStagesK;
  uint64_t* bar_emptyV = bar_fullV + C::kStagesV;
  uint64_t* bar_S = bar_emptyV + C::kStagesV;  // [NS] multicast: S of a tile computed
  uint64_t* bar_P = bar_S + NS;                // [NS] rank 0: P of a tile stored by both CTAs
  uint64_t* bar_O = bar_P + NS;                // [2] multicast: P(j).V(j) completes on O[j % 2]
  uint64_t* bar_Fin = bar_O + 2;               // multicast: last P.V done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::kStagesK; ++s) {
      mbar_init(&bar_fullK[s], 1);
      mbar_init(&bar_emptyK[s], 1);
    }
    for (int s = 0; s < C::kStagesV; ++s) {
      mbar_init(&bar_fullV[s], 1);
      mbar_init(&bar_emptyV[s], 1);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bar_S[i], 1);
      mbar_init(&bar_P[i], C::kPArrivals);
    }
    mbar_init(&bar_O[0], 1);
    mbar_init(&bar_O[1], 1);
    mbar_init(bar_Fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc_pair(tmem_slot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated before any use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= C::kSoftWarps) {
    // ======================= control warpgroup =======================
    if constexpr (C::NWG == 2) setmaxnreg_dec<C::kCtlRegs>();
    if (warp == C::kTmaWarp && n_kv > 0) {
      // =========================== TMA producer ===========================
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      if (rank == 0) mbar_arrive_expect_tx_e(bar_q, 2 * C::kQBytes);
      const uint32_t q_leader = mapa_shared(smem_u32(bar_q), 0);
#pragma unroll
      for (int p = 0; p < C::kPanels; ++p)
        tma_load_4d_pair_e(sQ + p * C::kQPanelBytes, &tm_q, q_leader, p * 64, hq, ext.qbase + q0, ext.bq);
      // the MMA warp takes K(j + kLook) before V(j)
      int jk = 0, jv = 0;
      bool aborted = false;
      while (jv < n_kv) {
        if (jk < n_kv && jk <= jv + C::kLook) {
          const int s = jk % C::kStagesK;
          const uint32_t ph = (uint32_t)(jk / C::kStagesK) & 1u;
          if (!mbar_wait_cl_warp(&bar_emptyK[s], ph ^ 1u, err, abort_flag)) { aborted = true; break; }
          if (rank == 0) mbar_arrive_expect_tx_e(&bar_fullK[s], 2 * C::kKStageBytes);
          const uint32_t full_leader = mapa_shared(smem_u32(&bar_fullK[s]), 0);
#pragma unroll
          for (int p = 0; p < C::kPanels; ++p)
            tma_load_4d_pair_e(sK + s * C::kKStageBytes + p * C::kKPanelBytes, &tm_k, full_leader, p * 64,
                               hk, tile_list_key(tl, jk) * BN + (int)rank * C::kKRows, b);
          ++jk;
          continue;
        }
        const int s = jv % C::kStagesV;
        const uint32_t ph = (uint32_t)(jv / C::kStagesV) & 1u;
        if (!mbar_wait_cl_warp(&bar_emptyV[s], ph ^ 1u, err, abort_flag)) { aborted = true; break; }
        if (rank == 0) mbar_arrive_expect_tx_e(&bar_fullV[s], 2 * C::kVStageBytes);
        const uint32_t full_leader = mapa_shared(smem_u32(&bar_fullV[s]), 0);
#pragma unroll
        for (int p = 0; p < C::kVPanels; ++p)
          tma_load_4d_pair_e(sV + s * C::kVStageBytes + p * C::kVPanelBytes, &tm_v, full_leader,
                             ((int)rank * C::kVPanels + p) * 64, hk, tile_list_key(tl, jv) * BN, b);
        ++jv;
      }
      if (aborted) {
        // The bytes of this CTA's copies complete on rank 0's barriers, which this
        // warp cannot wait on; give the copies already issued time to land
        // (about 1 ms) before the pair releases its shared memory.
        const long long t0 = clock64();
        while (clock64() - t0 < 2000000ll) {
        }
      }
    } else if (warp == C::kMmaWarp && rank == 0 && n_kv > 0) {
      // =========================== MMA issuer (rank 0) ===========================
      constexpr uint32_t idesc_s = idesc_bf16_f32(256, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(256, D, 0, 1);   // P (TMEM), V MN-major
      const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
      const uint64_t dk0 = smem_desc(smem_u32(sK), 16, 1024, kSwizzle128B);
      // V as the MN-major B operand: this CTA's 64-column panels are kVPanelBytes apart
      const uint64_t dv0 = smem_desc(smem_u32(sV), C::kVPanelBytes, 1024, kSwizzle128B);
      bool ok = mbar_wait_cl_warp(bar_q, 0, err, abort_flag);
      tc_fence_after();

      auto issue_s = [&](int j) {
        const uint64_t dk = dk0 + (uint64_t)(((j % C::kStagesK) * C::kKStageBytes) >> 4);
        const uint32_t d_tmem = tmem + C::s_col(j % NS);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t offq = (uint64_t)(((kk >> 2) * C::kQPanelBytes + (kk & 3) * 32) >> 4);
          const uint64_t offk = (uint64_t)(((kk >> 2) * C::kKPanelBytes + (kk & 3) * 32) >> 4);
          mma2_ss_e(d_tmem, dq + offq, dk + offk, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma2_commit_both_e(&bar_S[j % NS]);
      };
      auto issue_pv = [&](int j) -> bool {
        const int buf = j % NS;
        if (!mbar_wait_cl_warp(&bar_P[buf], (uint32_t)(j / NS) & 1u, err, abort_flag)) return false;
        tc_fence_after();
        const uint64_t dv = dv0 + (uint64_t)(((j % C::kStagesV) * C::kVStageBytes) >> 4);
        const uint32_t p_tmem = tmem + C::s_col(buf);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // keys [16kk, 16kk + 16): warpgroup g = 16kk / kCols stored them 8 (kk % (kCols / 16))
          // columns into its own S columns [g kCols, (g + 1) kCols)
          constexpr int kStepsPerWg = C::kCols / 16;
          const uint32_t a = p_tmem + C::kCols * (kk / kStepsPerWg) + 8 * (kk % kStepsPerWg);
          mma2_ts_e(tmem + C::o_col(), a, dv + (uint64_t)((kk * 2048) >> 4), idesc_o,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma2_commit_both_e(&bar_O[j & 1]);
        if (j == n_kv - 1) mma2_commit_both_e(bar_Fin);
        return true;
      };

      // prologue: S of the first kLook KV tiles
      for (int jj = 0; ok && jj < C::kLook && jj < n_kv; ++jj) {
        const int sk = jj % C::kStagesK;
        ok = mbar_wait_cl_warp(&bar_fullK[sk], (uint32_t)(jj / C::kStagesK) & 1u, err, abort_flag);
        tc_fence_after();
        if (ok) {
          issue_s(jj);
          mma2_commit_both_e(&bar_emptyK[sk]);
        }
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        // S(j + kLook) into the S buffer of P(j-1), read by P.V(j-1), issued before
        const int jn = j + C::kLook;
        if (jn < n_kv) {
          const int sn = jn % C::kStagesK;
          if (!mbar_wait_cl_warp(&bar_fullK[sn], (uint32_t)(jn / C::kStagesK) & 1u, err, abort_flag)) break;
          tc_fence_after();
          issue_s(jn);
          mma2_commit_both_e(&bar_emptyK[sn]);
        }
        const int s = j % C::kStagesV;
        if (!mbar_wait_cl_warp(&bar_fullV[s], (uint32_t)(j / C::kStagesV) & 1u, err, abort_flag)) break;
        tc_fence_after();
        if (!issue_pv(j)) break;
        mma2_commit_both_e(&bar_emptyV[s]);
      }
    }
  } else {
    // =========================== softmax warpgroups ===========================
    if constexpr (C::NWG == 2) setmaxnreg_inc<C::kSoftmaxRegs>();
    constexpr int KC = C::kCols, NWG = C::NWG;
    const int h = warp >> 2;         // key-column slice [h KC, (h + 1) KC) of every S tile
    const int wq = warp & 3;         // TMEM lane quarter
    const int r = wq * 32 + lane;    // row within the CTA's tile = TMEM lane
    const int qrow = q0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = scale * kLog2e;
    int row_bound = Skv;  // admissible keys of this row: [0, row_bound)
    if (causal) {
      const long long rb = (long long)qrow + off + 1;
      row_bound = (int)(rb < 0 ? 0 : (rb > Skv ? Skv : rb));
    }
    // with a window only [row_lo, row_bound) plus the sinks [0, n_sink); keys below the
    // window start of the CTA's last existing row need the mask (32-bit, clamped)
    auto clamp_key = [](long long x) { return (int)(x < -1 ? -1 : (x > 0x7FFFFFFF ? 0x7FFFFFFF : x)); };
    const int row_lo = WIN ? clamp_key((long long)qrow + off - window + 1) : -1;
    const int cta_lo_max =
        WIN ? clamp_key((long long)min(Sq, q0 + kPrefillTileM) - 1 + off - window + 1) : -1;
    float m_used = -INFINITY, l = 0.f, l_rnd = 0.f;
    bool ok = true;  // cleared by a failed wait; the loop still runs to the end so that
                     // both warpgroups meet at every exchange barrier

    for (int j = 0; j < n_kv; ++j) {
      const int buf = j % NS;
      ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait_cl(&bar_S[buf], (uint32_t)(j / NS) & 1u, err, abort_flag));
      tc_fence_after();
      const uint32_t s_addr = lane_addr + C::s_col(buf) + KC * h;
      uint32_t sr[KC];
      if (ok) {
#pragma unroll
        for (int c0 = 0; c0 < KC; c0 += 32) tmem_ld32(s_addr + c0, sr + c0);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int c = 0; c < KC; ++c) sr[c] = __float_as_uint(-INFINITY);
      }
      // mask: keys at or past row_bound (causal bound or Skv)
      const int key0 = tile_list_key(tl, j) * BN + KC * h;
      if (key0 + KC > kv_lo) {
        const int lim = row_bound - key0;
#pragma unroll
        for (int c = 0; c < KC; ++c)
          if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
      }
      if (WIN && key0 < cta_lo_max && key0 + KC > n_sink) {
#pragma unroll
        for (int c = 0; c < KC; ++c)
          if (key0 + c < row_lo && key0 + c >= n_sink) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx[4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
        mx[a] = max3f(__uint_as_float(sr[3 * a]), __uint_as_float(sr[3 * a + 1]), __uint_as_float(sr[3 * a + 2]));
#pragma unroll
      for (int c = 12; c < KC; c += 2)
        mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
      const float mh = fmaxf(max3f(mx[0], mx[1], mx[2]), mx[3]);
      // exchange the partial maxima with the other warpgroups (slot by tile parity);
      // every warpgroup takes the maximum in the same order, so all agree bit for bit
      float* xm = red + (j & 1) * (NWG * 128);
      xm[h * 128 + r] = mh;
      softmax_bar_sync<C::kSoftWarps * 32>();
      float mrow = xm[r];
#pragma unroll
      for (int g = 1; g < NWG; ++g) mrow = fmaxf(mrow, xm[g * 128 + r]);
      const float m_tile = mrow * sl2;
      const float m_new = fmaxf(m_used, m_tile);
      const bool need = m_new > m_used + kRescaleThreshold;
      if (__any_sync(0xFFFFFFFFu, need)) {
        const float corr = need ? ex2_approx(m_used - m_new) : 1.f;
        if (need) {
          l *= corr;
          l_rnd *= corr;
          m_used = m_new;
        }
        if (j > 0) {
          // O must hold P(j-1) V(j-1) before it is rescaled (this warpgroup's share of O)
          ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait_cl(&bar_O[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u,
                                                          err, abort_flag));
          tc_fence_after();
          if (ok) {
            const uint32_t o_addr = lane_addr + C::o_col() + h * (D / NWG);
#pragma unroll
            for (int c0 = 0; c0 < D / NWG; c0 += 32) {
              uint32_t ov[32];
              tmem_ld32(o_addr + c0, ov);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * corr);
              tmem_st32(o_addr + c0, ov);
            }
            tmem_wait_st();
          }
        }
      }
      const float msub = (m_used == -INFINITY) ? 0.f : m_used;
      const uint64_t sl2x2 = f2pack(sl2, sl2), nmx2 = f2pack(-msub, -msub);
      // two row sums: the exact one (for LSE) and one of the bf16-rounded weights the
      // P.V MMA uses (for O / l: consistent weights, so P rounding cancels for flat V)
      uint64_t lex2 = f2pack(0.f, 0.f);
      float lrd0 = 0.f, lrd1 = 0.f;
      uint32_t pk[KC / 2];
#pragma unroll
      for (int e = 0; e < KC / 2; ++e) {
        const uint64_t x2 = fma2(f2pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), sl2x2, nmx2);
        float x0, x1;
        f2unpack(x2, x0, x1);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        pk[e] = pack_bf16x2(p0, p1);
        lex2 = add2(lex2, f2pack(p0, p1));
        add_bf16x2_f32(pk[e], lrd0, lrd1);
      }
      {
        float a0, a1;
        f2unpack(lex2, a0, a1);
        l += a0 + a1;
        l_rnd += lrd0 + lrd1;
      }
      // P over the first KC / 2 of this warpgroup's S columns; then publish it to rank 0
      if (ok) {
        if constexpr (KC == 64) tmem_st32(s_addr, pk);
        else tmem_st16(s_addr, pk);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && ok) {
        if (rank == 0) mbar_arrive(&bar_P[buf]);
        else mbar_arrive_cluster(mapa_shared(smem_u32(&bar_P[buf]), 0));  // rank 0's barrier
      }
    }

    // ---- epilogue: combine the warpgroups' row sums, normalise O, store ----
    if (n_kv > 0) {
      ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait_cl(bar_Fin, 0, err, abort_flag));
      tc_fence_after();
    }
    float* xs = red + 2 * NWG * 128;  // [sum][h][row]
    xs[h * 128 + r] = l;
    xs[NWG * 128 + h * 128 + r] = l_rnd;
    softmax_bar_sync<C::kSoftWarps * 32>();
    float l_all = 0.f, lrnd_all = 0.f;
#pragma unroll
    for (int g = 0; g < NWG; ++g) {
      l_all += xs[g * 128 + r];
      lrnd_all += xs[NWG * 128 + g * 128 + r];
    }
    const bool load_o = ok && n_kv > 0;  // warp-uniform: tcgen05.ld is warp-collective
    const bool have = load_o && l_all > 0.f;
    const float inv_l = have ? 1.f / lrnd_all : 0.f;
    const bool row_ok = qrow < Sq;
    const uint32_t o_addr = lane_addr + C::o_col() + h * (D / NWG);
    const size_t orow = ((size_t)ext.bq * ext.rows + ext.qbase + (size_t)(row_ok ? qrow : 0)) * Hq + hq;
#pragma unroll
    for (int c0 = 0; c0 < D / NWG; c0 += 32) {
      uint32_t ov[32];
      if (load_o) {
        tmem_ld32(o_addr + c0, ov);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0u;
      }
      if (row_ok && ok) {
        const int col = h * (D / NWG) + c0;
        if (o_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(o_ptr) + orow * D + col);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(ov[8 * q4 + 0]) * inv_l, __uint_as_float(ov[8 * q4 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(ov[8 * q4 + 2]) * inv_l, __uint_as_float(ov[8 * q4 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(ov[8 * q4 + 4]) * inv_l, __uint_as_float(ov[8 * q4 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(ov[8 * q4 + 6]) * inv_l, __uint_as_float(ov[8 * q4 + 7]) * inv_l);
            dst[q4] = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(o_ptr) + orow * D + col);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            dst[q4] = make_float4(__uint_as_float(ov[4 * q4 + 0]) * inv_l, __uint_as_float(ov[4 * q4 + 1]) * inv_l,
                                  __uint_as_float(ov[4 * q4 + 2]) * inv_l, __uint_as_float(ov[4 * q4 + 3]) * inv_l);
          }
        }
      }
    }
    if (h == 0 && row_ok && ok) {
      lse_ptr[((size_t)ext.bq * Hq + hq) * ext.rows + ext.qbase + qrow] = have ? (m_used + log2f(l_all)) * kLn2 : -INFINITY;
    }
  }

  // ---- teardown: neither CTA frees TMEM or exits while the pair still works ----
  tc_fence_before();
  cluster_sync_all();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_pair_t(const PrefillArgs& a, cudaStream_t stream) {
  using C = PairCfg<D>;
  auto kern = a.window > 0 ? fmha_pair_kernel<D, true> : fmha_pair_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_blocks_q = (a.Sq + 2 * kPrefillTileM - 1) / (2 * kPrefillTileM);
  const long long units = (long long)n_blocks_q * a.Hq * a.B;
  if (units <= 0) return cudaSuccess;
  if (2 * units > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  kern<<<(unsigned)(2 * units), C::kThreads, C::kSmemBytes, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.o, a.lse, a.Hq, a.Hkv, a.Sq, a.Skv, a.causal, a.o_bf16, a.scale,
      a.Hq * a.B, a.err, a.cu_q, a.kv_lens, a.total_q, a.window, a.n_sink);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_pair(const PrefillArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 256: return launch_pair_t<256>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
