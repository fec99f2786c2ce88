// prefill_persist.cu -- persistent prefill FMHA for fixed-length batches (one query
// head per tile; head dims 64 and 128), causal or not.
//
// The arithmetic, the tiles and the warp roles are those of prefill.cu (two 128-row
// query tiles of one (batch, head) per work unit, S and P in TMEM, one MMA warp, the
// online softmax of "60 . r57 -- FA KV staging double buffering (REVERTED)",
// section 2.3, on the kernel shape of "STAGE_D.md -- FMHA Kernel Development",
// Architecture).  What differs is the schedule: one CTA per SM walks a sequence of
// units, so the work that surrounds a unit overlaps its neighbours instead of
// adding to it:
//   * Q of the next unit loads into a tile's Q buffer as soon as the tile's last
//     S MMA of the current unit has completed (a warp of its own issues it), and
//     the K and V rings run on across units, so the next unit's first tiles are in
//     shared memory when its first S MMAs are issued;
//   * O leaves through a staging tile of its own (not the Q buffer, which by then
//     holds the next unit's Q), which the two query tiles take in turn;
//   * in a causal unit the first query tile has one KV tile fewer than the second:
//     its softmax warpgroup writes its O during the second tile's last step.
// Units are dealt to the CTAs in waves, every other wave in reverse CTA order,
// over the heaviest-first unit order of the causal launch (the longest units go
// out first and each CTA gets a mix of long and short ones).
//
// Barrier phases run on across units: the K/V rings count items, the S, P and O
// barriers of a tile count its KV steps, its Q, Q-free and final barriers the units
// in which it has keys, and the staging barrier the turns.  (Counted by unit, the
// Q-free phases of key-less units were completed by the MMA warp without a wait, so
// it could run two phases ahead of the Q warp; and a tcgen05.commit issued before
// the CTA's first MMA was seen not to arrive.)
// Measured on the causal GQA workload (S = 3314, 28 heads): 86.7 -> 82.6 us against
// one CTA per unit.  Non-causal launches stay on prefill.cu, whose last wave runs as
// key halves (faster there: 193 against 209 us at d = 64, 222 against 236 at 128).
#include <algorithm>
#include <climits>
#include <cmath>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when m grows by > 2^8

template <int D>
struct PersistCfg {
  static constexpr int NQ = 2;                          // query tiles per unit
  static constexpr int BN = 128;                        // keys per KV tile
  static constexpr int kPanels = D / 64;                // 128-byte panels per row
  static constexpr int kPanelBytes = 128 * 128;         // one panel of 128 rows
  static constexpr int kTileBytes = kPanels * kPanelBytes;  // a Q tile, a K/V stage, the O staging tile
  static constexpr int kStagesK = D == 64 ? 4 : 2;
  static constexpr int kStagesV = D == 64 ? 4 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + NQ * kTileBytes;
  static constexpr int kVOff = kKOff + kStagesK * kTileBytes;
  static constexpr int kStgOff = kVOff + kStagesV * kTileBytes;
  static constexpr int kBarOff = kStgOff + kTileBytes;
  // barriers: Q[2], Qfree[2], fullK[SK], emptyK[SK], fullV[SV], emptyV[SV], S[2], P[2],
  // O[2], Fin[2], Stg
  static constexpr int kNumBars = 2 + 2 + 2 * kStagesK + 2 * kStagesV + 2 + 2 + 2 + 2 + 1;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  static constexpr int kThreads = 12 * 32;  // two softmax warpgroups + MMA, K, V and Q warps
  static constexpr int kMmaWarp = 8, kKWarp = 9, kVWarp = 10, kQWarp = 11;
  // register split as in prefill.cu: 8*32*208 + 4*32*80 = 63488 <= 384*168
  static constexpr int kLaunchRegs = 168;
  static constexpr int kSoftmaxRegs = 208;
  static constexpr int kCtlRegs = 80;
  static_assert((8 * kSoftmaxRegs + 4 * kCtlRegs) * 32 <= kThreads * kLaunchRegs, "register split");
  static constexpr uint32_t kTmemCols = 512;
  __host__ __device__ static constexpr uint32_t o_col(int t) { return (uint32_t)(t * D); }
  __host__ __device__ static constexpr uint32_t s_col(int t) { return (uint32_t)(NQ * D + t * BN); }
  static_assert(NQ * D + NQ * BN <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// One work unit: query block qb (rows [256 qb, 256 qb + 256)) of query head hq of
// batch b, and for each of its two query tiles the KV tiles it visits.
struct PUnit {
  int q0[2];     // first row of each query tile
  int n[2];      // KV tiles of each query tile (0: no admissible key, or past the end)
  int kv_lo[2];  // every row of the tile admits keys [0, kv_lo): later tiles need the mask
  int hq, hk, b;
};

__host__ __device__ __forceinline__ PUnit punit(int u, int Hq, int Hkv, int B, int Sq, int Skv, int causal) {
  const int n_blocks_q = (Sq + 2 * kPrefillTileM - 1) / (2 * kPrefillTileM);
  const int HB = Hq * B;
  // causal: heaviest query blocks first; non-causal: the query blocks of one head are
  // neighbours, so that head's K/V stay in L2 while they run
  const int qb = causal ? (n_blocks_q - 1 - u / HB) : (u % n_blocks_q);
  const int hb = causal ? (u % HB) : (u / n_blocks_q);
  PUnit p;
  p.hq = hb % Hq;
  p.b = hb / Hq;
  p.hk = p.hq / (Hq / Hkv);
  const long long off = (long long)Skv - Sq;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int q0 = qb * 2 * kPrefillTileM + t * kPrefillTileM;
    p.q0[t] = q0;
    if (q0 >= Sq) {
      p.n[t] = 0;
      p.kv_lo[t] = 0;
      continue;
    }
    int kv_hi = Skv, kv_lo = Skv;
    if (causal) {
      const int q_end = q0 + kPrefillTileM < Sq ? q0 + kPrefillTileM : Sq;
      const long long hi = (long long)(q_end - 1) + off + 1, lo = (long long)q0 + off + 1;
      kv_hi = (int)(hi < 0 ? 0 : (hi > Skv ? Skv : hi));
      kv_lo = (int)(lo < 0 ? 0 : (lo > Skv ? Skv : lo));
    }
    p.n[t] = (kv_hi + 128 - 1) / 128;
    p.kv_lo[t] = kv_lo;
  }
  return p;
}

// The k-th unit of CTA c, or -1 once the CTA has none left.  With a schedule
// (sched = offsets[grid + 1] followed by the unit lists) CTA c runs
// sched[grid + 1 + offsets[c] ...]; without one the units are dealt in waves of
// `grid`, every other wave in reverse CTA order.
__device__ __forceinline__ int unit_of(int k, int c, int grid, int units, const int* __restrict__ sched) {
  if (sched != nullptr) {
    const int i = __ldg(sched + c) + k;
    return i < __ldg(sched + c + 1) ? __ldg(sched + grid + 1 + i) : -1;
  }
  const long long u = (long long)k * grid + ((k & 1) ? grid - 1 - c : c);
  return u < units ? (int)u : -1;
}

template <int D>
__global__ void __launch_bounds__(PersistCfg<D>::kThreads, 1)
    fmha_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                           int o_tma, void* __restrict__ o_ptr, float* __restrict__ lse_ptr, int B, int Hq,
                           int Hkv, int Sq, int Skv, int causal, int o_bf16, float scale, int units,
                           const int* __restrict__ sched, uint32_t* err) {
  using C = PersistCfg<D>;
  constexpr int BN = C::BN;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = (int)blockIdx.x, grid = (int)gridDim.x;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  uint8_t* sStg = smem + C::kStgOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_q = bars;                          // [2] Q of a tile landed (one phase per unit)
  uint64_t* bar_qfree = bar_q + 2;                 // [2] the tile's last S MMA of a unit done
  uint64_t* bar_fullK = bar_qfree + 2;
  uint64_t* bar_emptyK = bar_fullK + C::kStagesK;
  uint64_t* bar_fullV = bar_emptyK + C::kStagesK;
  uint64_t* bar_emptyV = bar_fullV + C::kStagesV;
  uint64_t* bar_S = bar_emptyV + C::kStagesV;      // [2] one phase per KV step of the tile
  uint64_t* bar_P = bar_S + 2;                     // [2] one phase per KV step of the tile
  uint64_t* bar_O = bar_P + 2;                     // [2] one phase per P.V MMA group
  uint64_t* bar_Fin = bar_O + 2;                   // [2] the tile's last P.V of a unit done
  uint64_t* bar_stg = bar_Fin + 2;                 // the staging tile read out by its store
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_q[t], 1);
      mbar_init(&bar_qfree[t], 1);
      mbar_init(&bar_S[t], 1);
      mbar_init(&bar_P[t], 4);  // one arrive per softmax warp
      mbar_init(&bar_O[t], 1);
      mbar_init(&bar_Fin[t], 1);
    }
    for (int s = 0; s < C::kStagesK; ++s) {
      mbar_init(&bar_fullK[s], 1);
      mbar_init(&bar_emptyK[s], 1);
    }
    for (int s = 0; s < C::kStagesV; ++s) {
      mbar_init(&bar_fullV[s], 1);
      mbar_init(&bar_emptyV[s], 1);
    }
    mbar_init(bar_stg, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    // ======================= control warpgroup =======================
    setmaxnreg_dec<C::kCtlRegs>();
    if (warp == C::kQWarp) {
      // ----------------- Q producer: each unit's two Q tiles -----------------
      // A tile's Q and Q-free phases count the units in which it has keys (a tile
      // without rows or keys loads nothing and is not waited for).
      if (lane == 0) tma_prefetch_desc(&tm_q);
      bool ok = true;
      int m[2] = {0, 0};  // Q tiles loaded so far
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k, cta, grid, units, sched);
        if (u < 0) break;
        const PUnit p = punit(u, Hq, Hkv, B, Sq, Skv, causal);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || p.n[t] == 0) continue;
          // the tile's Q buffer is free once the last S MMA of its previous load is done
          if (m[t] > 0 && !(ok = mbar_wait_warp(&bar_qfree[t], (uint32_t)(m[t] - 1) & 1u, err, abort_flag)))
            break;
          mbar_arrive_expect_tx_e(&bar_q[t], C::kTileBytes);
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_5d_e(sQ + t * C::kTileBytes + pn * C::kPanelBytes, &tm_q, &bar_q[t], pn * 64, 0, p.hq,
                          p.q0[t], p.b);
          ++m[t];
        }
      }
    } else if (warp == C::kKWarp || warp == C::kVWarp) {
      // ----------------- K / V producers: one ring each, across units -----------------
      const bool is_k = warp == C::kKWarp;
      const int stages = is_k ? C::kStagesK : C::kStagesV;
      uint64_t* const full = is_k ? bar_fullK : bar_fullV;
      uint64_t* const empty = is_k ? bar_emptyK : bar_emptyV;
      uint8_t* const ring = is_k ? sK : sV;
      const CUtensorMap* const map = is_k ? &tm_k : &tm_v;
      if (lane == 0) tma_prefetch_desc(map);
      int g = 0;  // ring items issued
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k, cta, grid, units, sched);
        if (u < 0) break;
        const PUnit p = punit(u, Hq, Hkv, B, Sq, Skv, causal);
        const int n = max(p.n[0], p.n[1]);
        for (int j = 0; j < n; ++j, ++g) {
          const int s = g % stages;
          if (!(ok = mbar_wait_warp(&empty[s], ((uint32_t)(g / stages) & 1u) ^ 1u, err, abort_flag))) break;
          mbar_arrive_expect_tx_e(&full[s], C::kTileBytes);
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_4d_e(ring + s * C::kTileBytes + pn * C::kPanelBytes, map, &full[s], pn * 64, p.hk, j * BN, p.b);
        }
      }
      if (!ok) {
        // aborted: let the copies already issued land before shared memory is released
        for (int v = max(0, g - stages); v < g; ++v)
          mbar_wait(&full[v % stages], (uint32_t)(v / stages) & 1u, nullptr, nullptr, 100000000ull);
      }
    } else if (warp == C::kMmaWarp) {
      // ----------------- MMA issuer -----------------
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);   // P (TMEM), V MN-major
      uint64_t dq[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) dq[t] = smem_desc(smem_u32(sQ + t * C::kTileBytes), 16, 1024, kSwizzle128B);
      const uint64_t dk0 = smem_desc(smem_u32(sK), 16, 1024, kSwizzle128B);
      const uint64_t dv0 = smem_desc(smem_u32(sV), C::kPanelBytes, 1024, kSwizzle128B);
      int gk = 0, gv = 0;   // ring items consumed
      int J[2] = {0, 0};    // KV steps of each tile so far (S, P and O barrier phases)
      int mq[2] = {0, 0};   // units with keys of each tile so far (Q and Q-free phases)
      bool ok = true;
      // S_t = Q_t K(item gk)^T into tile t's S buffer
      auto issue_s = [&](int t) {
        const uint64_t dk = dk0 + (uint64_t)(((gk % C::kStagesK) * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * C::kPanelBytes + (kk & 3) * 32) >> 4);
          mma_ss_e(tmem + C::s_col(t), dq[t] + off, dk + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit_e(&bar_S[t]);
      };
      // O_t (+)= P_t V(item gv), P from tile t's S buffer; j: the tile's step in the unit
      auto issue_pv = [&](int t, int j, int n_t) -> bool {
        if (!mbar_wait_warp(&bar_P[t], (uint32_t)(J[t] + j) & 1u, err, abort_flag)) return false;
        tc_fence_after();
        const uint64_t dv = dv0 + (uint64_t)(((gv % C::kStagesV) * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)  // 16 keys = 8 TMEM columns of bf16 pairs, 2048 B of V
          mma_ts_e(tmem + C::o_col(t), tmem + C::s_col(t) + kk * 8, dv + (uint64_t)(kk * (2048 >> 4)), idesc_o,
                   (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_e(&bar_O[t]);
        if (j == n_t - 1) mma_commit_e(&bar_Fin[t]);
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k, cta, grid, units, sched);
        if (u < 0) break;
        const PUnit p = punit(u, Hq, Hkv, B, Sq, Skv, causal);
        const int n = max(p.n[0], p.n[1]);
        if (n > 0) {
          // this unit's Q tiles and its first K tile
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (ok && p.n[t] > 0) ok = mbar_wait_warp(&bar_q[t], (uint32_t)mq[t] & 1u, err, abort_flag);
          if (ok) ok = mbar_wait_warp(&bar_fullK[gk % C::kStagesK], (uint32_t)(gk / C::kStagesK) & 1u, err, abort_flag);
          tc_fence_after();
          if (!ok) break;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (p.n[t] > 0) {
              issue_s(t);
              if (p.n[t] == 1) mma_commit_e(&bar_qfree[t]);  // the tile's last S of the unit
            }
          }
          mma_commit_e(&bar_emptyK[gk % C::kStagesK]);
          ++gk;
          for (int j = 0; ok && j < n; ++j) {
            // V of step j, then per tile P.V(j) and S(j+1): S_t(j+1) overwrites P_t(j), so
            // it follows P_t(j).V(j); one tile's softmax runs while the other's MMAs do
            if (!(ok = mbar_wait_warp(&bar_fullV[gv % C::kStagesV], (uint32_t)(gv / C::kStagesV) & 1u, err,
                                      abort_flag)))
              break;
            tc_fence_after();
            bool k_ready = false;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (ok && j < p.n[t]) ok = issue_pv(t, j, p.n[t]);
              if (ok && j + 1 < p.n[t]) {
                if (!k_ready) {
                  ok = mbar_wait_warp(&bar_fullK[gk % C::kStagesK], (uint32_t)(gk / C::kStagesK) & 1u, err,
                                      abort_flag);
                  tc_fence_after();
                  k_ready = true;
                }
                if (ok) {
                  issue_s(t);
                  if (j + 2 == p.n[t]) mma_commit_e(&bar_qfree[t]);  // the tile's last S of the unit
                }
              }
            }
            if (!ok) break;
            if (k_ready) {
              mma_commit_e(&bar_emptyK[gk % C::kStagesK]);
              ++gk;
            }
            mma_commit_e(&bar_emptyV[gv % C::kStagesV]);
            ++gv;
          }
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) mq[t] += p.n[t] > 0 ? 1 : 0;
        J[0] += p.n[0];
        J[1] += p.n[1];
      }
    }
    // warp 11 (the Q producer) aside, the control warps are done
  } else {
    // =========================== softmax warpgroups ===========================
    setmaxnreg_inc<C::kSoftmaxRegs>();
    const int t = warp >> 2;         // query tile of this warpgroup
    const int wq = warp & 3;         // TMEM lane quarter
    const int r = wq * 32 + lane;    // row within the tile = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = scale * kLog2e;
    const long long pos_off = (long long)Skv - Sq;
    int J = 0;  // this tile's KV steps so far (S, P and O barrier phases)
    int F = 0;  // this tile's units with keys so far (final barrier phases)
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = unit_of(k, cta, grid, units, sched);
      if (u < 0) break;
      const PUnit p = punit(u, Hq, Hkv, B, Sq, Skv, causal);
      const int n_t = p.n[t];
      const int qrow = p.q0[t] + r;
      int row_bound = Skv;  // admissible keys of this row: [0, row_bound)
      if (causal) {
        const long long rb = (long long)qrow + pos_off + 1;
        row_bound = (int)(rb < 0 ? 0 : (rb > Skv ? Skv : rb));
      }
      float m_used = -INFINITY, l = 0.f, l_rnd = 0.f;

      for (int j = 0; j < n_t; ++j) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_S[t], (uint32_t)(J + j) & 1u, err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_addr = lane_addr + C::s_col(t);
        uint32_t sr[BN];
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) tmem_ld32(s_addr + c0, sr + c0);
        tmem_wait_ld();
        const int key0 = j * BN;
        if (key0 + BN > p.kv_lo[t]) {  // keys at or past the row's bound
          const int lim = row_bound - key0;
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
        }
        // row max: four independent chains of three-input max
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
            // O_t must hold P(j-1) V(j-1) before it is rescaled
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_O[t], (uint32_t)(J + j - 1) & 1u, err, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t o_addr = lane_addr + C::o_col(t);
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
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
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t sl2x2 = f2pack(sl2, sl2), nmx2 = f2pack(-msub, -msub);
        // two row sums: the exact one (for LSE) and one of the bf16-rounded weights the
        // P.V MMA uses (for O / l: consistent weights, so P rounding cancels for flat V)
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
            lex2 = add2(lex2, f2pack(p0, p1));
            add_bf16x2_f32(pk[e], lrd0, lrd1);
          }
          tmem_st16(s_addr + 16 * h, pk);  // P: bf16 pairs over the first BN/2 columns of S
        }
        {
          float a0, a1;
          f2unpack(lex2, a0, a1);
          l += a0 + a1;
          l_rnd += lrd0 + lrd1;
        }
        // publish P(j): the MMA warp reads it as the A operand of P.V
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_P[t]);
      }

      // ---- epilogue of this tile: O / l and LSE ----
      if (ok && n_t > 0) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_Fin[t], (uint32_t)F & 1u, err, abort_flag))) ok = false;
        tc_fence_after();
      }
      if (n_t > 0) ++F;
      const bool load_o = ok && n_t > 0;  // warp-uniform (tcgen05.ld is warp-collective)
      const bool have = load_o && l > 0.f;
      const float inv_l = have ? 1.f / l_rnd : 0.f;
      const bool row_ok = qrow < Sq;
      const uint32_t o_addr = lane_addr + C::o_col(t);
      auto load_o32 = [&](int c0, uint32_t* ov) {
        if (load_o) {
          tmem_ld32(o_addr + c0, ov);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = 0u;
        }
      };
      if (o_tma) {
        // bf16 O through the staging tile, which the two query tiles take in turn:
        // use e = 2k + t waits for use e - 1 to have been read out by its store
        const int e = 2 * k + t;
        if (e > 0 && !__all_sync(0xFFFFFFFFu, mbar_wait(bar_stg, (uint32_t)(e - 1) & 1u, err, abort_flag)))
          ok = false;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          load_o32(c0, ov);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(ov[8 * q4 + 0]) * inv_l, __uint_as_float(ov[8 * q4 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(ov[8 * q4 + 2]) * inv_l, __uint_as_float(ov[8 * q4 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(ov[8 * q4 + 4]) * inv_l, __uint_as_float(ov[8 * q4 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(ov[8 * q4 + 6]) * inv_l, __uint_as_float(ov[8 * q4 + 7]) * inv_l);
            const int chunk = (c0 >> 3) + q4;  // 16-byte chunk of the row
            const int pnl = chunk >> 3, cc = chunk & 7;
            *reinterpret_cast<uint4*>(sStg + pnl * C::kPanelBytes + r * 128 + ((cc ^ (r & 7)) << 4)) = w;
          }
        }
        fence_proxy_async_smem();
        // the warpgroup's rows are all in place (and every wait of theirs succeeded);
        // its four warps go on to the next unit, or stop, together
        const bool all_ok = bar_sync_and(1 + t, 128, ok);
        ok = all_ok;
        if ((threadIdx.x & 127) == 0) {
          if (all_ok && p.q0[t] < Sq) {  // a tile past the end stores nothing
#pragma unroll
            for (int pnl = 0; pnl < C::kPanels; ++pnl)
              tma_store_5d(&tm_o, sStg + pnl * C::kPanelBytes, pnl * 64, 0, p.hq, p.q0[t], p.b);
            tma_store_commit();
            tma_store_wait_read();  // the staging tile stays valid until the store has read it
          }
          mbar_arrive(bar_stg);  // always: the other tile's turn comes next
        }
      } else {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          load_o32(c0, ov);
          if (row_ok && ok) {
            const size_t orow = ((size_t)p.b * Sq + qrow) * Hq + p.hq;
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(o_ptr) + orow * D + c0);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(ov[4 * q4 + 0]) * inv_l, __uint_as_float(ov[4 * q4 + 1]) * inv_l,
                                    __uint_as_float(ov[4 * q4 + 2]) * inv_l, __uint_as_float(ov[4 * q4 + 3]) * inv_l);
          }
        }
      }
      if (!o_tma) ok = bar_sync_and(1 + t, 128, ok);  // the four warps go on, or stop, together
      if (row_ok && ok) {
        const float lse_v = have ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        lse_ptr[((size_t)p.b * Hq + p.hq) * Sq + qrow] = lse_v;
      }
      J += n_t;
    }
  }

  // ---- teardown: every role has finished with TMEM ----
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

int n_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// ---- the launch's unit schedule (host) ----
// A unit costs the KV steps of its longer query tile plus kUnitOverheadSteps for
// what surrounds it (Q load, the lone last step of the shorter tile's partner,
// the epilogue).  Dealt in waves, the causal units leave the CTAs unequal: their
// sizes come in a few coarse values (2, 4, ..., 26 steps for 3314 rows), and on
// the 28-head workload the most loaded of 152 CTAs carries 44 step-equivalents
// against a mean of 38.3 (at 2 steps of overhead per unit).  Best-fit decreasing
// -- each unit, largest first, goes to the fullest CTA it still fits into under a
// capacity, and the capacity is the smallest one for which every unit fits
// (bisection between the mean and the wave deal's maximum) -- packs them into 40.
// Each CTA then runs its units largest first.  Measured there (one GB300): wave
// deal 82.7-84.6 us; packed with an assumed overhead of 0, 1 and 2 steps per
// unit: 109.2, 88.7-89.8 and 78.5 us.  A fit of those times puts the real
// overhead near 2 steps; the packing assumes 3, which leaves the 28-head
// schedule's maximum at 40 if it is 2 and at 42 if it is 3.
constexpr long long kUnitOverheadSteps = 3;
// Launches with more units than this per CTA keep the wave deal: the imbalance it
// leaves is a small part of each CTA's share, and the packing's cost grows.
constexpr long long kMaxScheduledUnitsPerCta = 64;

bool pack_units(const std::vector<std::pair<long long, int>>& items, int grid, long long cap,
                std::vector<int>& cta_of) {
  std::set<std::pair<long long, int>> load;  // (load, CTA)
  for (int c = 0; c < grid; ++c) load.insert({0, c});
  for (const auto& it : items) {
    auto f = load.upper_bound({cap - it.first, INT_MAX});  // first CTA that would overflow
    if (f == load.begin()) return false;
    --f;  // the fullest CTA it fits into
    const std::pair<long long, int> b = *f;
    load.erase(f);
    load.insert({b.first + it.first, b.second});
    cta_of[it.second] = b.second;
  }
  return true;
}

}  // namespace

int build_prefill_schedule(int BH, int Sq, int Skv, int causal, int grid, std::vector<int>& sched) {
  sched.clear();
  const long long n_blocks_q = ((long long)Sq + 2 * kPrefillTileM - 1) / (2 * kPrefillTileM);
  const long long units = n_blocks_q * BH;
  if (BH < 1 || Sq < 0 || Skv < 0 || grid < 1 || units > 0x7FFFFFFFLL) return -1;
  if (units > kMaxScheduledUnitsPerCta * grid) return 0;
  std::vector<std::pair<long long, int>> items((size_t)units);  // (cost, unit)
  long long total = 0, biggest = 0;
  for (int u = 0; u < (int)units; ++u) {
    const PUnit p = punit(u, BH, BH, 1, Sq, Skv, causal);
    const long long w = (p.n[0] > p.n[1] ? p.n[0] : p.n[1]) + kUnitOverheadSteps;
    items[u] = {w, u};
    total += w;
    biggest = w > biggest ? w : biggest;
  }
  // the wave deal's most loaded CTA bounds the capacity from above
  std::vector<long long> wave(grid, 0);
  for (int c = 0; c < grid; ++c)
    for (int k = 0;; ++k) {
      const long long u = (long long)k * grid + ((k & 1) ? grid - 1 - c : c);
      if (u >= units) break;
      wave[c] += items[u].first;
    }
  long long hi = *std::max_element(wave.begin(), wave.end());
  long long lo = std::max((total + grid - 1) / grid, biggest);
  std::sort(items.begin(), items.end(), [](const auto& a, const auto& b) {
    return a.first != b.first ? a.first > b.first : a.second < b.second;
  });
  std::vector<int> cta_of((size_t)units, -1), best;
  if (!pack_units(items, grid, hi, cta_of)) return 0;  // keep the wave deal
  best = cta_of;
  while (lo < hi) {
    const long long mid = (lo + hi) / 2;
    if (pack_units(items, grid, mid, cta_of)) {
      best = cta_of;
      hi = mid;
    } else {
      lo = mid + 1;
    }
  }
  // offsets, then each CTA's units largest first (items are sorted that way)
  sched.assign((size_t)grid + 1 + (size_t)units, 0);
  for (int u = 0; u < (int)units; ++u) sched[best[u] + 1]++;
  for (int c = 0; c < grid; ++c) sched[c + 1] += sched[c];
  std::vector<int> fill(sched.begin(), sched.begin() + grid);
  for (const auto& it : items) sched[grid + 1 + fill[best[it.second]]++] = it.second;
  return (int)units;
}

namespace {

// Device copies of the schedules, one per (device, launch shape); built at a
// shape's first launch and kept until exit.  A launch that is being captured into
// a graph does not build one (the upload would break the capture): it takes the
// wave deal unless its shape was launched before.
struct SchedKey {
  int dev, BH, Sq, Skv, causal, grid;
  bool operator<(const SchedKey& o) const {
    return std::tie(dev, BH, Sq, Skv, causal, grid) < std::tie(o.dev, o.BH, o.Sq, o.Skv, o.causal, o.grid);
  }
};
constexpr size_t kMaxCachedSchedules = 256;

const int* device_schedule(const PrefillArgs& a, int grid, cudaStream_t stream) {
  static std::mutex mu;
  static std::map<SchedKey, int*> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  const SchedKey key{dev, a.B * a.Hq, a.Sq, a.Skv, a.causal, grid};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
  if (cache.size() >= kMaxCachedSchedules) return nullptr;
  std::vector<int> h;
  int* d = nullptr;
  if (build_prefill_schedule(key.BH, a.Sq, a.Skv, a.causal, grid, h) > 0) {
    if (cudaMalloc(&d, h.size() * sizeof(int)) != cudaSuccess) return nullptr;
    if (cudaMemcpy(d, h.data(), h.size() * sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaFree(d);
      return nullptr;
    }
  }
  cache[key] = d;  // nullptr: this shape keeps the wave deal
  return d;
}

template <int D>
cudaError_t launch_persist_t(const PrefillArgs& a, cudaStream_t stream) {
  using C = PersistCfg<D>;
  auto kern = fmha_persistent_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // the register split assumes the launch allocation it was sized for
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != C::kLaunchRegs) return cudaErrorInvalidConfiguration;
  const long long n_blocks_q = ((long long)a.Sq + 2 * kPrefillTileM - 1) / (2 * kPrefillTileM);
  const long long units = n_blocks_q * a.Hq * a.B;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const long long sms = n_sms();
  if (sms <= 0) return cudaErrorInvalidValue;
  const long long grid = units < sms ? units : sms;
  const int* sched = device_schedule(a, (int)grid, stream);
  kern<<<(unsigned)grid, C::kThreads, C::kSmemBytes, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.o_tma, a.o, a.lse, a.B, a.Hq, a.Hkv, a.Sq, a.Skv, a.causal, a.o_bf16,
      a.scale, (int)units, sched, a.err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_persistent(const PrefillArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_persist_t<64>(a, stream);
    case 128: return launch_persist_t<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
