// prefill_d512.cu -- exact attention forward (FMHA) for head dimension 512 on the
// 5th-generation tensor cores, on CTA pairs.
//
// Why a kernel of its own: tensor memory holds 512 columns of 128 lanes x 32
// bits.  With 128-row MMA tiles the fp32 O accumulator of a 512-wide head alone
// fills all of it and leaves no column for S; a CTA pair does not change that
// (each CTA still holds its 128 rows x every column of its accumulator).
// "STAGE_D.md -- FMHA Kernel Development", D1.4, meets the same head dimension
// as a shared-memory overflow and lists three ways out: tile Q along the head
// dimension, reuse buffers, split the GEMM's K dimension.  Here the head
// dimension is split everywhere it can be:
//   * O is computed in two column halves of 256, one after the other, by the
//     same CTAs (phase 0: columns [0, 256), phase 1: [256, 512)).  S = Q K^T is
//     recomputed in phase 1 -- 1.5x the tensor work of one pass, the price of
//     fitting O in tensor memory -- but the softmax of phase 1 needs no running
//     max: it reuses phase 0's final reference max, so it skips the max and the
//     O rescale;
//   * K and V stream through one ring of panel slots (the K-dimension split):
//     per KV tile the 8 panels of K (the S MMA's K dimension) and, per phase,
//     the V panels of that half's output columns;
//   * Q stays in shared memory for both phases (128 rows x 512 = 128 KB per
//     CTA, eight panels), so it is read from memory once.
// Tensor memory per CTA: the O half at columns [0, 256) and two S buffers at
// 256 and 384, so S of the next tile is computed while the softmax works on the
// current one.
//
// Both phases form one sequence of T = 2 n_kv tiles (tile jj: phase jj / n_kv,
// key tile jj % n_kv), issued as  S(0) S(1) { P(jj).V(jj)  S(jj + 2) }  so the
// pipeline runs through the phase boundary.  S(jj + 2) lands in S buffer jj % 2,
// over P(jj): it is issued after P(jj).V(jj), and MMAs from one thread execute
// in order.  The ring's items follow the same order: K(0) K(1) { V(jj) K(jj + 2) }.
//
// The arithmetic per phase is the one of prefill.cu (the online softmax of "60 .
// r57 -- FA KV staging double buffering (REVERTED)", section 2.3; O divided by
// the sum of the bf16-rounded weights it was accumulated with; LSE in natural
// log).  Phase 1 uses phase 0's final reference max m for every tile: its
// weights are exp(s - m) <= 2^8 (m lags the true maximum by at most the rescale
// threshold), and its own rounded-weight sum normalises its half of O.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when m grows by > 2^8

// A cluster of two CTAs takes 256 query rows of one (batch, query head), CTA r
// holding rows [128 r, 128 r + 128), and rank 0's MMA warp issues every MMA for
// both (cta_group::2, M = 256):
//   S = Q K^T     A = Q from each CTA's shared memory (its 128 rows), B = the
//                 128-key K tile split by keys: CTA r holds keys [64 r, 64 r + 64);
//   O += P V      A = P from each CTA's TMEM, B = a 128-column chunk of the
//                 phase's V half split by columns: CTA r holds columns
//                 [c 128 + 64 r, c 128 + 64 r + 64) of chunk c.
// Each CTA thus streams 96 KB per KV tile and phase, half of what one CTA doing
// the same MMA work alone would: a 96 KB ring holds twice the MMA time in flight.
// The ring has three 32 KB slots: a K item holds four 64-column panels of this
// CTA's 64 keys (two items per tile), a V item this CTA's panel of both
// 128-column chunks of the phase's half (one item per tile and phase).  Every
// item costs a round trip between the two SMs (its empty commit reaches the
// peer, the peer's bytes complete on rank 0's barrier), so fewer, larger items
// are faster: the same ring in 16 KB slots took 1.30x, in 8 KB slots 1.9x the
// time.  Every copy's bytes complete on rank 0's full barrier, armed by rank 0
// for both CTAs; MMA completions are multicast to the S, O, final and empty
// barriers of both CTAs; rank 1's softmax warps publish P with remote arrivals
// on rank 0's P barrier.  P.V(jj) completes on O barrier jj % 2, so that the
// previous use of the barrier a rescale waits on lies a whole P.V and S group
// back, even if the peer's copies of the arrivals are delivered out of order.
//
// Warp roles in each CTA (192 threads):
//   * warps 0-3  softmax (thread = TMEM lane = query row): read S, mask, keep
//       the running max m and sums (phase 0), write P (bf16) over the first half
//       of the S buffer, and at the end of each phase normalise that O half and
//       store it (and LSE, after phase 0);
//   * warp 4     TMEM allocation for the pair; in rank 0 also the MMA issuer (one
//       elected lane of the lock-step warp);
//   * warp 5     TMA producer: this CTA's Q tile once, then its share of every
//       ring item.
// A launch over at most 128 query rows leaves rank 1 without rows: it still
// takes its share of the MMAs (its Q tile reads as zeros past the end of the
// sequence) and stores nothing.
struct D512PairCfg {
  static constexpr int D = 512;
  static constexpr int BN = 128;                        // keys per KV tile (S columns)
  static constexpr int kPanels = D / 64;                // 64-column panels of a Q row
  static constexpr int kQPanelBytes = 128 * 128;        // 128 rows x 128 bytes, swizzled
  static constexpr int kKRows = BN / 2;                 // keys of a tile held by one CTA
  static constexpr int kKPanelBytes = kKRows * 128;     // 64 keys x 64 columns
  static constexpr int kSlotBytes = kD512PairSlotBytes; // one ring item
  static constexpr int kSlots = kD512PairRingBytes / kSlotBytes;
  // a K item: kKPanelsPerItem 64-column panels of this CTA's 64 keys
  static constexpr int kKPanelsPerItem = kSlotBytes / kKPanelBytes;
  static constexpr int kKItems = kPanels / kKPanelsPerItem;      // K items per tile
  // a V item: this CTA's 64-column panels of kVPanelsPerItem 128-column chunks,
  // kVRows keys of each
  static constexpr int kVRows = kD512PairVBoxRows;
  static constexpr int kVPanelBytes = kVRows * 128;
  static constexpr int kVPanelsPerItem = kSlotBytes / kVPanelBytes;
  static constexpr int kChunks = D / 2 / 128;                    // 128-column chunks of an O half
  static constexpr int kVItemsPerChunk = BN / kVRows;
  static constexpr int kVItems = kChunks * kVItemsPerChunk / kVPanelsPerItem;  // per tile and phase
  static_assert(kVPanelsPerItem >= 1 && kVItems * kVPanelsPerItem * kVPanelBytes == kChunks * BN * 128,
                "V items");
  static_assert(kKPanelsPerItem >= 1 && kKItems * kKPanelsPerItem == kPanels, "K items");
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kQOff + kPanels * kQPanelBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kSlotBytes;
  // barriers: Q, full[kSlots], empty[kSlots], S[2], P[2], O[2], Fin
  static constexpr int kNumBars = 1 + 2 * kSlots + 2 + 2 + 2 + 1;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;  // + alignment slack
  static constexpr int kThreads = 6 * 32;
  static constexpr int kMmaWarp = 4;
  static constexpr int kTmaWarp = 5;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCols = D / 2;             // one O half
  static constexpr uint32_t kPArrivals = 8;             // the softmax warps of both CTAs
  __host__ __device__ static constexpr uint32_t s_col(int buf) { return kOCols + (uint32_t)buf * BN; }
  static_assert(kOCols + 2 * BN <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(D512PairCfg::kThreads, 1)
    fmha_d512_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o_ptr,
                          float* __restrict__ lse_ptr, int B, int Hq, int Hkv, int Sq, int Skv, int causal,
                          int o_bf16, float scale, uint32_t* err) {
  using C = D512PairCfg;
  constexpr int BN = C::BN;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  // ---- work unit of the pair: 256 query rows of one (batch, query head) ----
  const int n_blocks_q = (Sq + 2 * kPrefillTileM - 1) / (2 * kPrefillTileM);
  const int HB = Hq * B;
  const int pair = (int)(blockIdx.x >> 1);
  // causal: heaviest query blocks first; non-causal: the query blocks of one head
  // are neighbours, so that head's K/V stay in L2 while they run
  const int qb = causal ? (n_blocks_q - 1 - pair / HB) : (pair % n_blocks_q);
  const int hb = causal ? (pair % HB) : (pair / n_blocks_q);
  const int hq = hb % Hq, b = hb / Hq;
  const int hk = hq / (Hq / Hkv);
  const int q0_pair = qb * 2 * kPrefillTileM;
  const int q0 = q0_pair + (int)rank * kPrefillTileM;  // this CTA's first query row
  const long long off = (long long)Skv - Sq;            // key position of query row i: i + off
  // KV tiles of the pair (both CTAs compute the same count) from its last row;
  // every row of this CTA admits [0, kv_lo)
  int kv_hi = Skv, kv_lo = Skv;
  if (causal) {
    const long long hi = (long long)(min(Sq, q0_pair + 2 * kPrefillTileM) - 1) + off + 1;
    const long long lo = (long long)q0 + off + 1;
    kv_hi = (int)(hi < 0 ? 0 : (hi > Skv ? Skv : hi));
    kv_lo = (int)(lo < 0 ? 0 : (lo > Skv ? Skv : lo));
  }
  const int n_kv = (kv_hi + BN - 1) / BN;
  const int T = 2 * n_kv;  // tiles of both phases

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* ring = smem + C::kRingOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_q = bars;                   // rank 0: both CTAs' Q bytes
  uint64_t* bar_full = bars + 1;            // rank 0: both CTAs' bytes of a ring item
  uint64_t* bar_empty = bar_full + C::kSlots;  // multicast: the item's MMAs completed
  uint64_t* bar_S = bar_empty + C::kSlots;  // [2] multicast: S of a tile computed in buffer b
  uint64_t* bar_P = bar_S + 2;              // [2] rank 0: P of a tile stored by both CTAs
  uint64_t* bar_O = bar_P + 2;              // [2] multicast: P(jj).V(jj) completes on O[jj % 2]
  uint64_t* bar_Fin = bar_O + 2;            // multicast: one phase per O half
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_S[i], 1);
      mbar_init(&bar_P[i], C::kPArrivals);
      mbar_init(&bar_O[i], 1);
    }
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

  if (warp == C::kTmaWarp) {
    // =========================== TMA producer (both CTAs) ===========================
    if (n_kv > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      if (rank == 0) mbar_arrive_expect_tx_e(bar_q, 2 * C::kPanels * C::kQPanelBytes);
      const uint32_t q_leader = mapa_shared(smem_u32(bar_q), 0);
#pragma unroll
      for (int p = 0; p < C::kPanels; ++p)
        tma_load_4d_pair_e(sQ + p * C::kQPanelBytes, &tm_q, q_leader, p * 64, hq, q0, b);
      int g = 0;  // ring items issued
      // wait for the next slot; rank 0 arms its full barrier for both CTAs' bytes
      auto slot = [&](uint8_t*& dst, uint32_t& full_leader) -> bool {
        const int s = g % C::kSlots;
        if (!mbar_wait_cl_warp(&bar_empty[s], ((uint32_t)(g / C::kSlots) & 1u) ^ 1u, err, abort_flag))
          return false;
        if (rank == 0) mbar_arrive_expect_tx_e(&bar_full[s], 2 * C::kSlotBytes);
        full_leader = mapa_shared(smem_u32(&bar_full[s]), 0);
        dst = ring + s * C::kSlotBytes;
        ++g;
        return true;
      };
      auto load_k = [&](int jj) -> bool {  // this CTA's 64 keys of tile jj
        const int key0 = (jj % n_kv) * BN + (int)rank * C::kKRows;
        for (int i = 0; i < C::kKItems; ++i) {
          uint8_t* dst;
          uint32_t fl;
          if (!slot(dst, fl)) return false;
#pragma unroll
          for (int p2 = 0; p2 < C::kKPanelsPerItem; ++p2)
            tma_load_4d_pair_e(dst + p2 * C::kKPanelBytes, &tm_k, fl, (i * C::kKPanelsPerItem + p2) * 64, hk,
                               key0, b);
        }
        return true;
      };
      auto load_v = [&](int jj) -> bool {  // this CTA's 64-column panel of each 128-column chunk
        const int ph = jj / n_kv, key0 = (jj % n_kv) * BN;
        for (int it = 0; it < C::kVItems; ++it) {
          const int c0 = (it / C::kVItemsPerChunk) * C::kVPanelsPerItem, kh = it % C::kVItemsPerChunk;
          uint8_t* dst;
          uint32_t fl;
          if (!slot(dst, fl)) return false;
#pragma unroll
          for (int pc = 0; pc < C::kVPanelsPerItem; ++pc)
            tma_load_4d_pair_e(dst + pc * C::kVPanelBytes, &tm_v, fl,
                               ph * (int)C::kOCols + (c0 + pc) * 128 + (int)rank * 64, hk, key0 + kh * C::kVRows, b);
        }
        return true;
      };
      bool ok = load_k(0) && load_k(1);
      for (int jj = 0; ok && jj < T; ++jj) ok = load_v(jj) && (jj + 2 >= T || load_k(jj + 2));
      if (!ok) {
        // The bytes of this CTA's copies complete on rank 0's barriers, which this
        // warp cannot wait on; give the copies already issued time to land
        // (about 1 ms) before the pair releases its shared memory.
        const long long t0 = clock64();
        while (clock64() - t0 < 2000000ll) {
        }
      }
    }
  } else if (warp == C::kMmaWarp) {
    // =========================== MMA issuer (rank 0) ===========================
    if (rank == 0 && n_kv > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(256, BN, 0, 0);   // Q, K both K-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(256, 128, 0, 1);  // P (TMEM), V MN-major
      const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
      const uint64_t dr = smem_desc(smem_u32(ring), 16, 1024, kSwizzle128B);
      // a V panel as the MN-major B operand: this CTA's 64 of the MMA's 128 columns,
      // one panel (the leading byte offset between panels is not used)
      const uint64_t dv0 = smem_desc(smem_u32(ring), C::kSlotBytes, 1024, kSwizzle128B);
      bool ok = mbar_wait_cl_warp(bar_q, 0, err, abort_flag);
      tc_fence_after();
      int g = 0;  // ring items consumed
      auto take = [&](int& s) -> bool {
        s = g % C::kSlots;
        if (!mbar_wait_cl_warp(&bar_full[s], (uint32_t)(g / C::kSlots) & 1u, err, abort_flag)) return false;
        tc_fence_after();
        return true;
      };
      // S(jj) = Q K(jj)^T into S buffer jj % 2: per K panel 4 K-steps of 16
      auto issue_s = [&](int jj) -> bool {
        const uint32_t d_tmem = tmem + C::s_col(jj & 1);
        for (int i = 0; i < C::kKItems; ++i) {
          int s;
          if (!take(s)) return false;
#pragma unroll
          for (int p2 = 0; p2 < C::kKPanelsPerItem; ++p2)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma2_ss_e(d_tmem, dq + (uint64_t)((((i * C::kKPanelsPerItem + p2) * C::kQPanelBytes) + kk * 32) >> 4),
                        dr + (uint64_t)((s * C::kSlotBytes + p2 * C::kKPanelBytes + kk * 32) >> 4), idesc_s,
                        (i | p2 | kk) ? 1u : 0u);
          mma2_commit_both_e(&bar_empty[s]);
          ++g;
        }
        mma2_commit_both_e(&bar_S[jj & 1]);
        return true;
      };
      // O_half[:, 128c, 128c + 128) += P(jj) V(jj)[:, chunk c]: P from the S buffer in TMEM
      auto issue_pv = [&](int jj) -> bool {
        const int j = jj % n_kv;
        if (!mbar_wait_cl_warp(&bar_P[jj & 1], (uint32_t)(jj >> 1) & 1u, err, abort_flag)) return false;
        tc_fence_after();
        const uint32_t p_tmem = tmem + C::s_col(jj & 1);
        for (int it = 0; it < C::kVItems; ++it) {
          const int c0 = (it / C::kVItemsPerChunk) * C::kVPanelsPerItem, kh = it % C::kVItemsPerChunk;
          int s;
          if (!take(s)) return false;
#pragma unroll
          for (int pc = 0; pc < C::kVPanelsPerItem; ++pc)
#pragma unroll
            for (int kk = 0; kk < C::kVRows / 16; ++kk) {  // 16 keys = 8 TMEM columns of bf16 pairs, 2 KB of V
              const int kg = kh * (C::kVRows / 16) + kk;   // 16-key step within the tile
              mma2_ts_e(tmem + (uint32_t)((c0 + pc) * 128), p_tmem + kg * 8,
                        dv0 + (uint64_t)((s * C::kSlotBytes + pc * C::kVPanelBytes + kk * 2048) >> 4), idesc_o,
                        (j > 0 || kg > 0) ? 1u : 0u);
            }
          mma2_commit_both_e(&bar_empty[s]);
          ++g;
        }
        mma2_commit_both_e(&bar_O[jj & 1]);
        if (j == n_kv - 1) mma2_commit_both_e(bar_Fin);
        return true;
      };
      ok = ok && issue_s(0) && issue_s(1);
      for (int jj = 0; ok && jj < T; ++jj) ok = issue_pv(jj) && (jj + 2 >= T || issue_s(jj + 2));
    }
  } else {
    // =========================== softmax warpgroup (both CTAs) ===========================
    const int r = warp * 32 + lane;  // row within this CTA's tile = TMEM lane
    const int qrow = q0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = scale * kLog2e;
    int row_bound = Skv;  // admissible keys of this row: [0, row_bound)
    if (causal) {
      const long long rb = (long long)qrow + off + 1;
      row_bound = (int)(rb < 0 ? 0 : (rb > Skv ? Skv : rb));
    }
    const bool row_ok = qrow < Sq;
    float m_used = -INFINITY, l = 0.f, l_rnd = 0.f;
    bool ok = true;

    // normalise O half `ph` of this row and store it (and LSE after phase 0)
    auto epilogue = [&](int ph) {
      if (ok && n_kv > 0) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_cl(bar_Fin, (uint32_t)ph, err, abort_flag))) ok = false;
        tc_fence_after();
      }
      const bool load_o = ok && n_kv > 0;  // warp-uniform (tcgen05.ld is warp-collective)
      const float inv_l = (load_o && l_rnd > 0.f) ? 1.f / l_rnd : 0.f;
      const size_t orow = ((size_t)b * Sq + (size_t)(row_ok ? qrow : 0)) * Hq + hq;
      const int col0 = ph * (int)C::kOCols;
#pragma unroll 1
      for (int c0 = 0; c0 < (int)C::kOCols; c0 += 32) {
        uint32_t ov[32];
        if (load_o) {
          tmem_ld32(lane_addr + (uint32_t)c0, ov);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = 0u;
        }
        if (!(row_ok && ok)) continue;
        if (o_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(o_ptr) + orow * C::D + col0 + c0);
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
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(o_ptr) + orow * C::D + col0 + c0);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4] = make_float4(__uint_as_float(ov[4 * q4 + 0]) * inv_l, __uint_as_float(ov[4 * q4 + 1]) * inv_l,
                                  __uint_as_float(ov[4 * q4 + 2]) * inv_l, __uint_as_float(ov[4 * q4 + 3]) * inv_l);
        }
      }
      if (ph == 0 && row_ok && ok) {
        const bool have = n_kv > 0 && l > 0.f;  // at least one admissible key
        lse_ptr[((size_t)b * Hq + hq) * Sq + qrow] = have ? (m_used + log2f(l)) * kLn2 : -INFINITY;
      }
    };

    for (int jj = 0; jj < T; ++jj) {
      const int ph = jj >= n_kv ? 1 : 0;
      const int j = jj - ph * n_kv;
      const int buf = jj & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_cl(&bar_S[buf], (uint32_t)(jj >> 1) & 1u, err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_addr = lane_addr + C::s_col(buf);
      uint32_t sr[BN];
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) tmem_ld32(s_addr + c0, sr + c0);
      tmem_wait_ld();
      const int key0 = j * BN;
      if (key0 + BN > kv_lo) {  // keys at or past the row's bound
        const int lim = row_bound - key0;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
      }
      if (ph == 0) {
        float mx[4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
          mx[a] = max3f(__uint_as_float(sr[3 * a]), __uint_as_float(sr[3 * a + 1]), __uint_as_float(sr[3 * a + 2]));
#pragma unroll
        for (int c = 12; c < BN; c += 2)
          mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
        const float m_tile = fmaxf(max3f(mx[0], mx[1], mx[2]), mx[3]) * sl2;
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
            // O must hold P(jj-1) V(jj-1) before it is rescaled
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_cl(&bar_O[(jj - 1) & 1], (uint32_t)((jj - 1) >> 1) & 1u, err,
                                                      abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < (int)C::kOCols; c0 += 32) {
              uint32_t ov[32];
              tmem_ld32(lane_addr + (uint32_t)c0, ov);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * corr);
              tmem_st32(lane_addr + (uint32_t)c0, ov);
            }
            tmem_wait_st();
          }
        }
      }
      const float msub = (m_used == -INFINITY) ? 0.f : m_used;
      const uint64_t sl2x2 = f2pack(sl2, sl2), nmx2 = f2pack(-msub, -msub);
      uint64_t lex2 = f2pack(0.f, 0.f);
      float lrd0 = 0.f, lrd1 = 0.f;
#pragma unroll
      for (int h = 0; h < BN / 32; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t x2 = fma2(f2pack(__uint_as_float(sr[32 * h + 2 * e]),
                                          __uint_as_float(sr[32 * h + 2 * e + 1])), sl2x2, nmx2);
          float x0, x1;
          f2unpack(x2, x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          pk[e] = pack_bf16x2(p0, p1);
          if (ph == 0) lex2 = add2(lex2, f2pack(p0, p1));
          add_bf16x2_f32(pk[e], lrd0, lrd1);
        }
        tmem_st16(s_addr + 16 * h, pk);  // P: bf16 pairs over the first BN/2 columns of S
      }
      if (ph == 0) {
        float a0, a1;
        f2unpack(lex2, a0, a1);
        l += a0 + a1;
      }
      l_rnd += lrd0 + lrd1;
      // publish P(jj) to rank 0's MMA warp
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&bar_P[buf]);
        else mbar_arrive_cluster(mapa_shared(smem_u32(&bar_P[buf]), 0));
      }
      if (j == n_kv - 1) {
        epilogue(ph);
        l_rnd = 0.f;  // phase 1 sums its own rounded weights
      }
    }
    if (n_kv == 0) {  // no admissible key for any row of the pair: O = 0, LSE = -inf
      epilogue(0);
      epilogue(1);
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

}  // namespace

cudaError_t launch_prefill_d512(const PrefillArgs& a, cudaStream_t stream) {
  using C = D512PairCfg;
  cudaError_t e = cudaFuncSetAttribute(fmha_d512_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long n_blocks_q = ((long long)a.Sq + 2 * kPrefillTileM - 1) / (2 * kPrefillTileM);
  const long long units = n_blocks_q * a.Hq * a.B;
  if (units <= 0) return cudaSuccess;
  if (2 * units > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  fmha_d512_pair_kernel<<<(unsigned)(2 * units), C::kThreads, C::kSmemBytes, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.o, a.lse, a.B, a.Hq, a.Hkv, a.Sq, a.Skv, a.causal, a.o_bf16, a.scale, a.err);
  return cudaGetLastError();
}

}  // namespace attn
