// prefill.cu -- exact attention forward (FMHA) on the 5th-generation tensor cores.
//
// Per CTA: NQ query tiles of 128 rows of one (batch, query head), streamed
// against 128-row K/V tiles of the matching KV head.  Warp roles:
//   * warps 0 .. 4*NQ-1  softmax warpgroups, one per query tile (thread = row):
//       read S from TMEM, apply the causal / length mask, keep the running
//       row max m and row sum l, rescale O in TMEM when m grows by more than
//       2^8, write P (bf16) back into TMEM over S, and finally normalise O and
//       store O and LSE;
//   * warp 4*NQ       MMA issuer (one thread): S = Q K^T and O += P V with
//       tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in TMEM; P is the A
//       operand straight from TMEM);
//   * warp 4*NQ+1     TMA producer (one thread): Q once, then a ring of K and
//       V stages, each 128 rows x d, 128-byte swizzled.
//
// The algorithm is the online softmax of "60 . r57 -- FA KV staging double
// buffering (REVERTED)", section 2.3 (at every KV tile boundary
// m_new = max(m_old, tile_max) and O is rescaled by exp(m_old - m_new)), with
// the kernel shape of "STAGE_D.md -- FMHA Kernel Development", Architecture
// (TMA warp / MMA warp / softmax warps), TMEM Layout and P Staging Paths (P
// kept in TMEM as the A operand of the P.V MMA).  What differs from that page:
// O is normalised in-kernel (each thread owns one TMEM lane = one row, so the
// TMEM round trip is a plain 32x32b load/store with matching shapes), LSE is in
// natural-log units, and the O rescale is skipped while the running max has
// grown by at most 2^8 (the final O / l uses the same stale max in numerator
// and denominator, so the result is unchanged up to rounding).
//
// TMEM columns (512 allocated, 128 lanes):
//   NQ = 2 (d <= 128):  tile t: S/P at t*(128 + d) ... one S buffer per tile
//   NQ = 1 (d == 256):  S buffers at 0 and 128, O at 256
// Scheduling (MMA issue order) keeps the tensor pipe busy while the softmax
// warps work:  NQ = 2:  PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) ...
//              NQ = 1:  S(j+1) PV(j) ...  (two S buffers)
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when m grows by > 2^8

template <int D>
struct PrefillCfg {
  static constexpr int NQ = (D <= 128) ? 2 : 1;            // query tiles per CTA
  static constexpr int NS = (NQ == 2) ? 1 : 2;             // S buffers per query tile
  static constexpr int kPanels = D / 64;                   // 128-byte panels per row
  static constexpr int kPanelBytes = 128 * 128;            // 128 rows x 128 bytes
  static constexpr int kTileBytes = kPanels * kPanelBytes; // one 128 x d bf16 tile
#ifndef ATTN_PREFILL_KSTAGES
  static constexpr int kStagesK = (D == 64) ? 4 : (D == 128 ? 2 : 1);  // K ring depth
#else
  static constexpr int kStagesK = ATTN_PREFILL_KSTAGES;
#endif
#ifndef ATTN_PREFILL_VSTAGES
  static constexpr int kStagesV = (D == 64) ? 4 : (D == 128 ? 2 : 1);  // V ring depth
#else
  static constexpr int kStagesV = ATTN_PREFILL_VSTAGES;
#endif
  static constexpr int kQOff = 0;
  static constexpr int kKOff = NQ * kTileBytes;
  static constexpr int kVOff = kKOff + kStagesK * kTileBytes;
  static constexpr int kBarOff = kVOff + kStagesV * kTileBytes;
  // barriers: fullQ, fullK[SK], emptyK[SK], fullV[SV], emptyV[SV], S[NQ][NS], P[NQ], O[NQ], Fin[NQ]
  static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + NQ * NS + 3 * NQ;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  // NQ softmax warpgroups + one control warpgroup (MMA warp, TMA warp, two spare warps).
  static constexpr int kThreads = (4 * NQ + 4) * 32;
  static constexpr int kMmaWarp = 4 * NQ;
  static constexpr int kTmaWarp = 4 * NQ + 1;
  // Register split (NQ == 2 only; 12 warps launch with 168 registers each):
  // the control warpgroup drops to kCtlRegs, the softmax warpgroups grow to
  // kSoftmaxRegs: 8*32*208 + 4*32*80 = 63488 <= 384*168 = 64512 (the launch
  // total), and per SM sub-partition 2*208 + 80 = 496 <= 512 registers per lane.
  static constexpr int kLaunchRegs = 168;
  static constexpr int kSoftmaxRegs = 208;
  static constexpr int kCtlRegs = 80;
  static_assert(NQ != 2 || (4 * NQ * kSoftmaxRegs + 4 * kCtlRegs) * 32 <= kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
  static constexpr uint32_t kTmemCols = 512;
  // TMEM column of S buffer `buf` of tile t, and of O of tile t
  __host__ __device__ static constexpr uint32_t s_col(int t, int buf) {
    return NQ == 2 ? (uint32_t)(t * (128 + D)) : (uint32_t)(buf * 128);
  }
  __host__ __device__ static constexpr uint32_t o_col(int t) {
    return NQ == 2 ? (uint32_t)(t * (128 + D) + 128) : 256u;
  }
  static_assert(NQ * (NS * 128 + D) <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Rows of query tile t that exist, and its KV extent.
struct TileInfo {
  int q0;      // first query row of the tile
  int n_kv;    // KV tiles to visit (0: no admissible key for any existing row)
  int kv_lo;   // every existing row of the tile admits keys [0, kv_lo): tiles past it need a mask
};

__device__ __forceinline__ TileInfo tile_info(int q0, int Sq, int Skv, int causal) {
  TileInfo ti;
  ti.q0 = q0;
  if (q0 >= Sq) {
    ti.n_kv = 0;
    ti.kv_lo = 0;
    return ti;
  }
  const int q_last = min(Sq, q0 + kPrefillTileM) - 1;
  int kv_hi = Skv, kv_lo = Skv;
  if (causal) {
    const long long off = (long long)Skv - Sq;
    long long hi = (long long)q_last + off + 1, lo = (long long)q0 + off + 1;
    kv_hi = (int)(hi < 0 ? 0 : (hi > Skv ? Skv : hi));
    kv_lo = (int)(lo < 0 ? 0 : (lo > Skv ? Skv : lo));
  }
  ti.n_kv = (kv_hi + kPrefillTileN - 1) / kPrefillTileN;
  ti.kv_lo = kv_lo;
  return ti;
}

template <int D>
__global__ void __launch_bounds__(PrefillCfg<D>::kThreads, 1)
    fmha_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o_ptr,
                    float* __restrict__ lse_ptr, int Hq, int Hkv, int Sq, int Skv, int causal,
                    int o_bf16, float scale, int n_units_per_head_batch, uint32_t* err) {
  using C = PrefillCfg<D>;
  constexpr int NQ = C::NQ, NS = C::NS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work unit: longest causal work first ----
  const int HB = n_units_per_head_batch;  // Hq * B
  const int n_blocks_q = (Sq + NQ * kPrefillTileM - 1) / (NQ * kPrefillTileM);
  const int u = blockIdx.x;
  const int qb = causal ? (n_blocks_q - 1 - u / HB) : (u / HB);
  const int hb = u % HB;
  const int hq = hb % Hq, b = hb / Hq;
  const int hk = hq / (Hq / Hkv);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_q = bars;
  uint64_t* bar_fullK = bars + 1;
  uint64_t* bar_emptyK = bar_fullK + C::kStagesK;
  uint64_t* bar_fullV = bar_emptyK + C::kStagesK;
  uint64_t* bar_emptyV = bar_fullV + C::kStagesV;
  uint64_t* bar_S = bar_emptyV + C::kStagesV;  // [NQ][NS]
  uint64_t* bar_P = bar_S + NQ * NS;          // [NQ]
  uint64_t* bar_O = bar_P + NQ;               // [NQ] one phase per P.V MMA group
  uint64_t* bar_Fin = bar_O + NQ;             // [NQ] last P.V done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  TileInfo ti[NQ];
#pragma unroll
  for (int t = 0; t < NQ; ++t) ti[t] = tile_info(qb * NQ * kPrefillTileM + t * kPrefillTileM, Sq, Skv, causal);
  int n_kv = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) n_kv = max(n_kv, ti[t].n_kv);

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
    for (int i = 0; i < NQ * NS; ++i) mbar_init(&bar_S[i], 1);
    for (int t = 0; t < NQ; ++t) {
      mbar_init(&bar_P[t], 4);  // one arrive per softmax warp
      mbar_init(&bar_O[t], 1);
      mbar_init(&bar_Fin[t], 1);
    }
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

  if (warp >= 4 * NQ) {
    // ======================= control warpgroup =======================
    if constexpr (NQ == 2) setmaxnreg_dec<C::kCtlRegs>();  // whole warpgroup, same instruction
  if (warp == C::kTmaWarp) {
    // =========================== TMA producer ===========================
    // The whole warp runs the loop; one elected lane issues each copy.
    if (n_kv > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      uint32_t qbytes = 0;
#pragma unroll
      for (int t = 0; t < NQ; ++t)
        if (ti[t].n_kv > 0) qbytes += C::kTileBytes;
      mbar_arrive_expect_tx_e(bar_q, qbytes);
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        if (ti[t].n_kv > 0) {
#pragma unroll
          for (int p = 0; p < C::kPanels; ++p)
            tma_load_4d_e(sQ + t * C::kTileBytes + p * C::kPanelBytes, &tm_q, bar_q, p * 64, hq,
                          ti[t].q0, b);
        }
      }
      // K(j) and V(j) alternate; each ring has its own depth
      int jk = 0, jv = 0;
      bool aborted = false;
      while (jv < n_kv) {
        if (jk < n_kv && jk <= jv) {
          const int s = jk % C::kStagesK;
          const uint32_t ph = (uint32_t)(jk / C::kStagesK) & 1u;
          if (!mbar_wait_warp(&bar_emptyK[s], ph ^ 1u, err, abort_flag)) { aborted = true; break; }
          mbar_arrive_expect_tx_e(&bar_fullK[s], C::kTileBytes);
#pragma unroll
          for (int p = 0; p < C::kPanels; ++p)
            tma_load_4d_e(sK + s * C::kTileBytes + p * C::kPanelBytes, &tm_k, &bar_fullK[s], p * 64,
                          hk, jk * kPrefillTileN, b);
          ++jk;
          continue;
        }
        const int s = jv % C::kStagesV;
        const uint32_t ph = (uint32_t)(jv / C::kStagesV) & 1u;
        if (!mbar_wait_warp(&bar_emptyV[s], ph ^ 1u, err, abort_flag)) { aborted = true; break; }
        mbar_arrive_expect_tx_e(&bar_fullV[s], C::kTileBytes);
#pragma unroll
        for (int p = 0; p < C::kPanels; ++p)
          tma_load_4d_e(sV + s * C::kTileBytes + p * C::kPanelBytes, &tm_v, &bar_fullV[s], p * 64,
                        hk, jv * kPrefillTileN, b);
        ++jv;
      }
      if (aborted) {
        // let the copies already issued land before shared memory is released
        for (int u2 = max(0, jk - C::kStagesK); u2 < jk; ++u2)
          mbar_wait(&bar_fullK[u2 % C::kStagesK], (uint32_t)(u2 / C::kStagesK) & 1u, nullptr, nullptr,
                    100000000ull);
        for (int u2 = max(0, jv - C::kStagesV); u2 < jv; ++u2)
          mbar_wait(&bar_fullV[u2 % C::kStagesV], (uint32_t)(u2 / C::kStagesV) & 1u, nullptr, nullptr,
                    100000000ull);
      }
    }
  } else if (warp == C::kMmaWarp) {
    // =========================== MMA issuer ===========================
    // The whole warp runs the loop with warp-uniform descriptors; one elected
    // lane issues each tcgen05.mma / commit.
    if (n_kv > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);  // Q, K both K-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);    // P (TMEM), V MN-major
      constexpr uint64_t kTileDesc = (uint64_t)(C::kTileBytes >> 4);  // descriptor step per tile
      uint64_t dq[NQ];
#pragma unroll
      for (int t = 0; t < NQ; ++t)
        dq[t] = smem_desc(smem_u32(sQ + t * C::kTileBytes), 16, 1024, kSwizzle128B);
      const uint64_t dk0 = smem_desc(smem_u32(sK), 16, 1024, kSwizzle128B);
      const uint64_t dv0 = smem_desc(smem_u32(sV), C::kPanelBytes, 1024, kSwizzle128B);
      bool ok = mbar_wait_warp(bar_q, 0, err, abort_flag);
      tc_fence_after();

      // S_t(j) = Q_t K_j^T into S buffer `buf`
      auto issue_s = [&](int t, int j, int buf) {
        const uint64_t dk = dk0 + (uint64_t)(j % C::kStagesK) * kTileDesc;
        const uint32_t d_tmem = tmem + C::s_col(t, buf);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * C::kPanelBytes + (kk & 3) * 32) >> 4);
          mma_ss_e(d_tmem, dq[t] + off, dk + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit_e(&bar_S[t * NS + buf]);
      };
      // O_t += P_t(j) V_j, P read from TMEM over S buffer `buf`
      auto issue_pv = [&](int t, int j, int buf) {
        const uint64_t dv = dv0 + (uint64_t)(j % C::kStagesV) * kTileDesc;
        const uint32_t p_tmem = tmem + C::s_col(t, buf);
        const uint32_t d_tmem = tmem + C::o_col(t);
#pragma unroll
        for (int kk = 0; kk < kPrefillTileN / 16; ++kk)
          mma_ts_e(d_tmem, p_tmem + kk * 8, dv + (uint64_t)(kk * (2048 >> 4)), idesc_o,
                   (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_e(&bar_O[t]);
        if (j == ti[t].n_kv - 1) mma_commit_e(&bar_Fin[t]);
      };

      if (ok) {
        // prologue: S of the first KV tile (and the second one with two S buffers)
        ok = mbar_wait_warp(&bar_fullK[0], 0, err, abort_flag);
        tc_fence_after();
        if (ok) {
#pragma unroll
          for (int t = 0; t < NQ; ++t)
            if (ti[t].n_kv > 0) issue_s(t, 0, 0);
          mma_commit_e(&bar_emptyK[0]);
        }
        if constexpr (NQ == 1) {
          if (ok && n_kv > 1) {
            ok = mbar_wait_warp(&bar_fullK[1 % C::kStagesK], (uint32_t)(1 / C::kStagesK) & 1u, err,
                                abort_flag);
            tc_fence_after();
            if (ok) {
              issue_s(0, 1, 1);
              mma_commit_e(&bar_emptyK[1 % C::kStagesK]);
            }
          }
        }
        for (int j = 0; ok && j < n_kv; ++j) {
          const int s = j % C::kStagesV;
          const uint32_t ph = (uint32_t)(j / C::kStagesV) & 1u;
          if (!mbar_wait_warp(&bar_fullV[s], ph, err, abort_flag)) break;
          tc_fence_after();
          if constexpr (NQ == 2) {
            const int jn = j + 1;
            bool k_ready = false;
#pragma unroll
            for (int t = 0; t < NQ; ++t) {
              if (j < ti[t].n_kv) {
                if (!mbar_wait_warp(&bar_P[t], (uint32_t)j & 1u, err, abort_flag)) { ok = false; break; }
                tc_fence_after();
                issue_pv(t, j, 0);
              }
              if (jn < ti[t].n_kv) {
                if (!k_ready) {
                  const int sn = jn % C::kStagesK;
                  if (!mbar_wait_warp(&bar_fullK[sn], (uint32_t)(jn / C::kStagesK) & 1u, err, abort_flag)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                  k_ready = true;
                }
                issue_s(t, jn, 0);
              }
            }
            if (!ok) break;
            if (k_ready) mma_commit_e(&bar_emptyK[jn % C::kStagesK]);
            mma_commit_e(&bar_emptyV[s]);
          } else {
            // two S buffers: S(j+1) was issued one iteration ahead; issue S(j+2) after PV(j)
            if (!mbar_wait_warp(&bar_P[0], (uint32_t)j & 1u, err, abort_flag)) break;
            tc_fence_after();
            issue_pv(0, j, j & 1);
            // release V(j) before waiting on K(j+2): the producer loads V(j+1) ahead of K(j+2)
            mma_commit_e(&bar_emptyV[s]);
            const int jn = j + 2;
            if (jn < n_kv) {
              const int sn = jn % C::kStagesK;
              if (!mbar_wait_warp(&bar_fullK[sn], (uint32_t)(jn / C::kStagesK) & 1u, err, abort_flag)) break;
              tc_fence_after();
              issue_s(0, jn, jn & 1);
              mma_commit_e(&bar_emptyK[sn]);
            }
          }
        }
      }
    }
  }
  } else {
    // =========================== softmax warpgroups ===========================
    if constexpr (NQ == 2) setmaxnreg_inc<C::kSoftmaxRegs>();
    const int t = warp >> 2;         // query tile of this warpgroup
    const int wq = warp & 3;         // TMEM lane quarter
    const int r = wq * 32 + lane;    // row within the tile = TMEM lane
    const TileInfo my = ti[t];
    const int qrow = my.q0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = scale * kLog2e;
    // admissible keys of this row: [0, row_bound)
    int row_bound = Skv;
    if (causal) {
      const long long rb = (long long)qrow + ((long long)Skv - Sq) + 1;
      row_bound = (int)(rb < 0 ? 0 : (rb > Skv ? Skv : rb));
    }
    float m_used = -INFINITY, l = 0.f, l_rnd = 0.f;
    bool ok = true;

    for (int j = 0; j < my.n_kv; ++j) {
      const int buf = (NS == 1) ? 0 : (j & 1);
      const uint32_t sph = (NS == 1) ? ((uint32_t)j & 1u) : ((uint32_t)(j >> 1) & 1u);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_S[t * NS + buf], sph, err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_addr = lane_addr + C::s_col(t, buf);
      uint32_t sr[128];
      tmem_ld32(s_addr + 0, sr + 0);
      tmem_ld32(s_addr + 32, sr + 32);
      tmem_ld32(s_addr + 64, sr + 64);
      tmem_ld32(s_addr + 96, sr + 96);
      tmem_wait_ld();
      // mask: keys at or past row_bound (causal bound or Skv)
      if ((j + 1) * kPrefillTileN > my.kv_lo) {
        const int lim = row_bound - j * kPrefillTileN;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
      }
      // row max: four independent chains of three-input max
      float mx[4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
        mx[a] = max3f(__uint_as_float(sr[3 * a]), __uint_as_float(sr[3 * a + 1]), __uint_as_float(sr[3 * a + 2]));
#pragma unroll
      for (int c = 12; c < 128; c += 2)
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
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_O[t], (uint32_t)(j - 1) & 1u, err, abort_flag))) {
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
      uint64_t lex2 = f2pack(0.f, 0.f), lrd2 = f2pack(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
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
          lrd2 = add2(lrd2, f2pack(__uint_as_float(pk[e] << 16), __uint_as_float(pk[e] & 0xFFFF0000u)));
        }
        tmem_st16(s_addr + 16 * h, pk);  // P: bf16 pairs over the first 64 columns of S
      }
      {
        float a0, a1, b0, b1;
        f2unpack(lex2, a0, a1);
        f2unpack(lrd2, b0, b1);
        l += a0 + a1;
        l_rnd += b0 + b1;
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_P[t]);
    }

    // ---- epilogue: O / l and LSE ----
    if (ok && my.n_kv > 0) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_Fin[t], 0, err, abort_flag))) ok = false;
      tc_fence_after();
    }
    // warp-uniform: tcgen05.ld below is a warp-collective instruction
    const bool load_o = ok && my.n_kv > 0;
    const bool have = load_o && l > 0.f;  // per row: at least one admissible key
    const float inv_l = have ? 1.f / l_rnd : 0.f;
    const bool row_ok = qrow < Sq;
    const uint32_t o_addr = lane_addr + C::o_col(t);
    const size_t orow = ((size_t)b * Sq + (size_t)(row_ok ? qrow : 0)) * Hq + hq;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t ov[32];
      if (load_o) {
        tmem_ld32(o_addr + c0, ov);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0u;
      }
      if (row_ok && ok) {
        if (o_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(o_ptr) + orow * D + c0);
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
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(o_ptr) + orow * D + c0);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            dst[q4] = make_float4(__uint_as_float(ov[4 * q4 + 0]) * inv_l, __uint_as_float(ov[4 * q4 + 1]) * inv_l,
                                  __uint_as_float(ov[4 * q4 + 2]) * inv_l, __uint_as_float(ov[4 * q4 + 3]) * inv_l);
          }
        }
      }
    }
    if (row_ok && ok) {
      lse_ptr[((size_t)b * Hq + hq) * Sq + qrow] = have ? (m_used + log2f(l)) * kLn2 : -INFINITY;
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

// Skv == 0: no key at all, O = 0 and LSE = -inf for every row.
__global__ void fill_empty_kernel(void* o, float* lse, size_t n_o, size_t n_lse, int o_bf16) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_o; i += stride) {
    if (o_bf16) reinterpret_cast<uint16_t*>(o)[i] = 0;
    else reinterpret_cast<float*>(o)[i] = 0.f;
  }
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_lse; i += stride)
    lse[i] = -INFINITY;
}

template <int D>
cudaError_t launch_prefill_t(const PrefillArgs& a, cudaStream_t stream) {
  using C = PrefillCfg<D>;
  auto kern = fmha_fwd_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_blocks_q = (a.Sq + C::NQ * kPrefillTileM - 1) / (C::NQ * kPrefillTileM);
  const long long units = (long long)n_blocks_q * a.Hq * a.B;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  kern<<<(unsigned)units, C::kThreads, C::kSmemBytes, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.o, a.lse, a.Hq, a.Hkv, a.Sq, a.Skv, a.causal, a.o_bf16, a.scale,
      a.Hq * a.B, a.err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_prefill_t<64>(a, stream);
    case 128: return launch_prefill_t<128>(a, stream);
    case 256: return launch_prefill_t<256>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefill_empty_kv(const PrefillArgs& a, cudaStream_t stream) {
  const size_t n_o = (size_t)a.B * a.Sq * a.Hq * a.d;
  const size_t n_lse = (size_t)a.B * a.Hq * a.Sq;
  if (n_o == 0) return cudaSuccess;
  fill_empty_kernel<<<1024, 256, 0, stream>>>(a.o, a.lse, n_o, n_lse, a.o_bf16);
  return cudaGetLastError();
}

}  // namespace attn
