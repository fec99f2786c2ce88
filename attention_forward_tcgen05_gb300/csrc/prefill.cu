// prefill.cu -- exact attention forward (FMHA) on the 5th-generation tensor cores,
// one CTA per query block: used for head dims 64 and 128 (head dim 256 runs on
// CTA pairs, prefill_pair.cu; the d = 256 configuration below is kept for
// comparison and is not launched).
//
// Per CTA: NQ query tiles of 128 rows of one (batch, query head), streamed
// against K/V tiles of BN = 128 rows of the matching KV head, which arrive by
// TMA in stages of 128 rows (the kernel also runs 64-row tiles, two per stage,
// with one TMA box per 128 rows: the copy engine's cost grows with the number
// of boxes much more than with their size).  Warp roles:
//   * warps 0 .. 4*NQ-1  softmax warpgroups, one per query tile (thread = row):
//       read S from TMEM, apply the causal / length mask, keep the running
//       row max m and row sum l, rescale O in TMEM when m grows by more than
//       2^8, write P (bf16) back into TMEM over S, and finally normalise O and
//       store O and LSE;
//   * warp 4*NQ       MMA issuer: S = Q K^T and O += P V with tcgen05.mma
//       (kind::f16, bf16 in, fp32 accumulate in TMEM; P is the A operand
//       straight from TMEM);
//   * warps 4*NQ+1, 4*NQ+2  TMA producers: Q once and then a ring of K stages,
//       and a ring of V stages, each 128 rows x d, 128-byte swizzled; the two
//       rings fill independently.
// The MMA and TMA warps run their loops as whole warps (warp-uniform
// descriptors); one elected lane issues each instruction.
//
// The algorithm is the online softmax of "60 . r57 -- FA KV staging double
// buffering (REVERTED)", section 2.3 (at every KV tile boundary
// m_new = max(m_old, tile_max) and O is rescaled by exp(m_old - m_new)), with
// the kernel shape of "STAGE_D.md -- FMHA Kernel Development", Architecture
// (TMA warp / MMA warp / softmax warps), TMEM Layout and P Staging Paths (P
// kept in TMEM as the A operand of the P.V MMA).  What differs from that page:
// O is normalised in-kernel (each thread owns one TMEM lane = one row, so the
// TMEM round trip is a plain 32x32b load/store with matching shapes), LSE is in
// natural-log units, the O rescale is skipped while the running max has grown
// by at most 2^8 (the final O / l uses the same stale max in numerator and
// denominator, so the result is unchanged up to rounding), and for d = 256
// the query tile has two S buffers.
//
// TMEM columns (512 allocated, 128 lanes): O of tile t at t*d, then the S
// buffers, BN = 128 columns each:  d = 256: O_0 S_00 S_01;  d <= 128:
// O_0 O_1 S_0 S_1 (one S buffer per tile).  With two S buffers the MMA warp computes
// S(j+1) = Q K(j+1)^T while the softmax warps work on S(j); the issue order
// per KV tile j is  S_0(j+1) [S_1(j+1)] P_0(j).V(j) [P_1(j).V(j)],  so the
// tensor pipe is never idle waiting for a softmax pass.  P(j) lives in the S
// buffer of tile j, and S(j+2) overwrites it only after P(j).V(j) (issued
// earlier, executed in order) has read it.  With one S buffer per tile (d <=
// 128: two S buffers per tile would leave room for 64-key tiles only, which
// need twice the MMA instructions per key, each re-reading Q from shared
// memory; measured slower) the order
// is  P_0(j).V(j) S_0(j+1) P_1(j).V(j) S_1(j+1):  S_t(j+1) follows P_t(j).V(j),
// and each tile's softmax overlaps the other tile's MMAs.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when m grows by > 2^8

// H: the key-halves layout (both query tiles read one Q tile, the freed Q space
// deepens the K ring for keys streamed from HBM)
template <int D, bool H = false>
struct PrefillCfg {
  static constexpr int NQ = (D <= 128) ? 2 : 1;            // query tiles per CTA
  static constexpr int NS = (D == 256) ? 2 : 1;            // S buffers per query tile
  // rows of a K / V tile (S has BN columns): TMEM holds NQ O tiles of d columns
  // and NQ*NS S buffers of BN columns
  static constexpr int BN = (NQ * D + NQ * NS * 128 <= 512) ? 128 : 64;
  static constexpr int kStageRows = kPrefillKVStageRows;   // rows of a TMA-loaded K / V stage
  static constexpr int kSub = kStageRows / BN;             // KV tiles per stage
  static constexpr int kPanels = D / 64;                   // 128-byte panels per row
  static constexpr int kQPanelBytes = kPrefillTileM * 128; // one panel of a Q tile
  static constexpr int kKVPanelBytes = kStageRows * 128;   // one panel of a K / V stage
  static constexpr int kSubBytes = BN * 128;               // offset of tile h of a stage in a panel
  static constexpr int kQTileBytes = kPanels * kQPanelBytes;
  static constexpr int kKVStageBytes = kPanels * kKVPanelBytes;
  static constexpr int kStagesK = (D == 64) ? (H ? 5 : 4) : (D == 128 ? (H ? 3 : 2) : 1);  // K ring depth
  static constexpr int kStagesV = (D == 64) ? 4 : (D == 128 ? (H ? 2 : 3) : 1);  // V ring depth
  static constexpr int kQTiles = H ? 1 : NQ;               // Q tiles in shared memory
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQTiles * kQTileBytes;
  static constexpr int kVOff = kKOff + kStagesK * kKVStageBytes;
  static constexpr int kBarOff = kVOff + kStagesV * kKVStageBytes;
  // barriers: fullQ, fullK[SK], emptyK[SK], fullV[SV], emptyV[SV], S[NQ][NS],
  // P[NQ][NS], O[NQ], Fin[NQ].  S and P have one barrier per S buffer, so each
  // is at most one phase ahead of the warp that waits on it.
  static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + 2 * NQ * NS + 2 * NQ;
  // merge of the two key halves of a decode unit: per row (m, l, l_rnd, ok), fp32
  // (key-halves layout only)
  static constexpr int kMergeOff = kBarOff + kNumBars * 8 + 16;
  static constexpr int kMergeBytes = H ? 128 * 4 * 4 : 0;
  static constexpr int kSmemBytes = kMergeOff + kMergeBytes + 1024;
  // NQ softmax warpgroups + one control warpgroup (MMA warp, K and V TMA warps, one
  // spare warp).
  static constexpr int kThreads = (4 * NQ + 4) * 32;
  static constexpr int kMmaWarp = 4 * NQ;
  static constexpr int kTmaWarp = 4 * NQ + 1;  // K producer; kTmaWarp + 1: V producer
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
  __host__ __device__ static constexpr uint32_t o_col(int t) { return (uint32_t)(t * D); }
  __host__ __device__ static constexpr uint32_t s_col(int t, int buf) {
    return (uint32_t)(NQ * D + (t * NS + buf) * BN);
  }
  static_assert(NQ * D + NQ * NS * BN <= 512, "TMEM budget");
  static_assert(BN % 32 == 0 && BN <= 128, "S is read in 32-column loads; P.V has K = BN");
  static_assert(kStageRows % BN == 0 && kSubBytes % 1024 == 0, "tiles start on a swizzle atom");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Rows of query tile t that exist, and its KV extent.
struct TileInfo {
  int q0;      // first query row of the tile
  int n_kv;    // KV tiles to visit (0: no admissible key for any existing row)
  int kv_lo;   // every existing row of the tile admits keys [0, kv_lo): tiles past it need a mask
};

// q0: first row of the tile; Sr: rows of the sequence (Sq positions x G heads);
// the causal bound of a row follows its position row / G.  Keys at or past kend
// (the end of a key split; Skv without one) are not admitted.
template <int BN>
__device__ __forceinline__ TileInfo tile_info(int q0, int Sr, int Sq, int G, int Skv, int causal,
                                              int kend) {
  TileInfo ti;
  ti.q0 = q0;
  if (q0 >= Sr) {
    ti.n_kv = 0;
    ti.kv_lo = 0;
    return ti;
  }
  const int q_last = (min(Sr, q0 + kPrefillTileM) - 1) / G;  // positions
  const int q_first = q0 / G;
  int kv_hi = Skv, kv_lo = Skv;
  if (causal) {
    const long long off = (long long)Skv - Sq;
    long long hi = (long long)q_last + off + 1, lo = (long long)q_first + off + 1;
    kv_hi = (int)(hi < 0 ? 0 : (hi > Skv ? Skv : hi));
    kv_lo = (int)(lo < 0 ? 0 : (lo > Skv ? Skv : lo));
  }
  kv_hi = min(kv_hi, kend);
  ti.n_kv = (kv_hi + BN - 1) / BN;
  ti.kv_lo = min(kv_lo, kend);
  return ti;
}

// WIN: causal sliding window with attention sinks (window, n_sink); without it
// both are ignored and the tile list is every KV tile.  SPLIT: key splits with
// decode partials (n_splits, split_min, part_o, part_lse); without it they are ignored.
// HALVES (one query position per sequence, its G <= 128 head rows in one tile):
// both query tiles hold the same rows and take the two halves of the unit's keys,
// so their S -> softmax -> P.V chains overlap; the halves merge in the epilogue.
template <int D, bool WIN, bool SPLIT, bool HALVES>
__global__ void __launch_bounds__(PrefillCfg<D, HALVES>::kThreads, 1)
    fmha_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    int o_tma, void* __restrict__ o_ptr,
                    float* __restrict__ lse_ptr, int Hq, int Hkv, int Sq_max, int Skv_max, int causal,
                    int o_bf16, float scale, int n_units_per_head_batch, uint32_t* err,
                    const int* __restrict__ cu_q, const int* __restrict__ kv_lens, int total_q,
                    int window, int n_sink, int pack, int n_splits, int split_min,
                    float* __restrict__ part_o, float* __restrict__ part_lse, int unit0,
                    int row_halves) {
  using C = PrefillCfg<D, HALVES>;
  constexpr int NQ = C::NQ, NS = C::NS, BN = C::BN;
  static_assert(C::kSub == 1, "a KV stage is one tile (the sliding-window tile list maps tiles, not stages)");
  static_assert(!HALVES || (NQ == 2 && NS == 1 && !WIN), "key halves: two query tiles, no window");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work unit ----
  // A unit is NQ query tiles of one head group: G = pack query heads (of one KV
  // head) folded into the tile rows, row r = (position r / G, head r % G).
  const int G = pack;
  const int Hu = Hq / G;                  // head groups
  const int HB = n_units_per_head_batch;  // Hu * B
  const int n_blocks_q = (Sq_max * G + NQ * kPrefillTileM - 1) / (NQ * kPrefillTileM);
  // key splits (one-token decode only): unit = (query block, split, head group, batch)
  const int NSPL = SPLIT ? n_splits : 1;
  // CTA -> unit: this launch covers units [unit0, ...); with row halves (key-halves
  // kernel) CTA pairs share a unit, each taking 128 rows of its query block
  const int u = unit0 + ((HALVES && row_halves) ? (int)(blockIdx.x >> 1) : (int)blockIdx.x);
  const int rh = (HALVES && row_halves) ? (int)(blockIdx.x & 1) : 0;
  // causal: heaviest query blocks first; non-causal: the query blocks of one head
  // are neighbours, so that head's K/V stay in L2 while they run
  const int qb = causal ? (n_blocks_q - 1 - u / (HB * NSPL)) : (u % n_blocks_q);
  const int sp = causal ? (u % (HB * NSPL)) / HB : 0;
  const int hb = causal ? u % HB : u / n_blocks_q;
  const int hu = hb % Hu, b = hb / Hu;
  const int hk = (hu * G) / (Hq / Hkv);
  // this sequence's query positions and keys (fixed-length or packed varlen batch)
  const SeqExtent ext = seq_extent(b, Sq_max, Skv_max, cu_q, kv_lens, total_q);
  const int Sq = ext.Sq, Skv = ext.Skv;
  const int Sr = Sq * G;  // tile rows of this sequence
  // keys [klo, khi) of this unit: split sp of the sequence's keys (the split rule of
  // the decode partials: chunk = max(ceil(Skv / n_splits), split_min)), or all of them
  int klo = 0, khi = Skv;
  if (SPLIT) {
    const int chunk = max((Skv + NSPL - 1) / NSPL, split_min);
    const long long lo = (long long)sp * chunk;
    klo = (int)min((long long)Skv, lo);
    khi = (int)min((long long)Skv, lo + chunk);
  }

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
  uint64_t* bar_S = bar_emptyV + C::kStagesV;  // [NQ][NS] S of a KV tile computed
  uint64_t* bar_P = bar_S + NQ * NS;           // [NQ][NS] P of a KV tile stored
  uint64_t* bar_O = bar_P + NQ * NS;           // [NQ] one phase per P.V MMA group
  uint64_t* bar_Fin = bar_O + NQ;              // [NQ] last P.V done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  TileInfo ti[NQ];
#pragma unroll
  for (int t = 0; t < NQ; ++t)
    ti[t] = tile_info<BN>(qb * NQ * kPrefillTileM + (t + rh) * kPrefillTileM, Sr, Sq, G, Skv, causal, khi);
  int n_kv = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) n_kv = max(n_kv, ti[t].n_kv);
  // the loops below run over a list of KV tiles (list index j, key tile
  // tile_list_key(tl, j)): with a sliding window the sink tiles and the window's
  // tiles, with a key split the tiles from the split's first one, else every tile
  const long long pos_off = (long long)Skv - Sq;  // key position of query row i: i + pos_off
  const TileList tl = WIN ? tile_list((long long)(ti[0].q0 / G) + pos_off, n_kv, window, n_sink, Skv, BN)
                          : (SPLIT ? TileList{0, klo / BN} : TileList{0x7FFFFFFF, 0});
#pragma unroll
  for (int t = 0; t < NQ; ++t) ti[t].n_kv = klo < khi ? tile_list_len(tl, ti[t].n_kv) : 0;
  n_kv = klo < khi ? tile_list_len(tl, n_kv) : 0;
  // key halves: tile 0 takes list entries [0, n0), tile 1 (the same rows) [n0, n)
  // (with a key split, of the split's tiles); the K/V rings run over items
  // i = (step i / 2, tile i % 2)
  int n_items = n_kv, n0 = n_kv;
  if constexpr (HALVES) {
    const int n = ti[0].n_kv;
    n0 = (n + 1) / 2;
    ti[1] = ti[0];
    ti[1].n_kv = n - n0;
    ti[0].n_kv = n0;
    n_kv = n0;
    n_items = n;
  }
  // key tile of ring item i (the TMA order) and of list entry j of query tile t
  auto item_key = [&](int i) -> int {
    if constexpr (HALVES) return tile_list_key(tl, (i & 1) ? n0 + (i >> 1) : (i >> 1));
    return tile_list_key(tl, i);
  };

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
    for (int i = 0; i < NQ * NS; ++i) {
      mbar_init(&bar_S[i], 1);
      mbar_init(&bar_P[i], 4);  // one arrive per softmax warp
    }
    for (int t = 0; t < NQ; ++t) {
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
  if (warp == C::kTmaWarp || warp == C::kTmaWarp + 1) {
    // =========================== TMA producers ===========================
    // Warp kTmaWarp loads Q once and then the K ring, warp kTmaWarp + 1 the V ring.
    // The rings fill independently: a stage is requested as soon as it is free,
    // so a V stage never waits behind a K stage that is still in use (with one
    // producer issuing K(j+1) before V(j), a wait for a K slot held up the V load
    // the MMA warp needed next).
    if (n_kv > 0) {
      const bool is_k = warp == C::kTmaWarp;
      if (lane == 0) {
        if (is_k) {
          tma_prefetch_desc(&tm_q);
          tma_prefetch_desc(&tm_k);
        } else {
          tma_prefetch_desc(&tm_v);
        }
      }
      if (is_k) {
        // a Q box holds 128 / G whole positions of G head rows: all 128 rows of the
        // tile when G divides 128, else the first G * floor(128 / G) (one-token decode
        // only, whose single position is in tile 0; the rows below are never read
        // out)
        const uint32_t q_box_bytes = (uint32_t)(G * (kPrefillTileM / G)) * 128u * C::kPanels;
        uint32_t qbytes = 0;
#pragma unroll
        for (int t = 0; t < C::kQTiles; ++t)
          if (ti[t].n_kv > 0) qbytes += q_box_bytes;
        mbar_arrive_expect_tx_e(bar_q, qbytes);
#pragma unroll
        for (int t = 0; t < C::kQTiles; ++t) {
          if (ti[t].n_kv > 0) {
#pragma unroll
            for (int p = 0; p < C::kPanels; ++p)
              tma_load_5d_e(sQ + t * C::kQTileBytes + p * C::kQPanelBytes, &tm_q, bar_q, p * 64, 0, hu,
                            ext.qbase + ti[t].q0 / G, ext.bq);
          }
        }
      }
      // stages of kSub KV tiles (ring items with key halves), in the order the MMA
      // warp consumes them
      const int n_st = (n_items + C::kSub - 1) / C::kSub;
      const int stages = is_k ? C::kStagesK : C::kStagesV;
      uint64_t* const full = is_k ? bar_fullK : bar_fullV;
      uint64_t* const empty = is_k ? bar_emptyK : bar_emptyV;
      uint8_t* const ring = is_k ? sK : sV;
      const CUtensorMap* const map = is_k ? &tm_k : &tm_v;
      int u = 0;
      for (; u < n_st; ++u) {
        const int s = u % stages;
        const uint32_t ph = (uint32_t)(u / stages) & 1u;
        if (!mbar_wait_warp(&empty[s], ph ^ 1u, err, abort_flag)) break;
        mbar_arrive_expect_tx_e(&full[s], C::kKVStageBytes);
#pragma unroll
        for (int p = 0; p < C::kPanels; ++p)
          tma_load_4d_e(ring + s * C::kKVStageBytes + p * C::kKVPanelBytes, map, &full[s], p * 64, hk,
                        item_key(u) * C::kStageRows, b);
      }
      if (u < n_st) {
        // aborted: let the copies already issued land before shared memory is released
        for (int u2 = max(0, u - stages); u2 < u; ++u2)
          mbar_wait(&full[u2 % stages], (uint32_t)(u2 / stages) & 1u, nullptr, nullptr, 100000000ull);
      }
    }
  } else if (warp == C::kMmaWarp) {
    // =========================== MMA issuer ===========================
    if (n_kv > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);   // P (TMEM), V MN-major
      // descriptor start of KV tile j: its stage, then its rows within each panel
      auto kv_tile_desc = [&](uint64_t d0, int j, int stages) -> uint64_t {
        const int off = ((j / C::kSub) % stages) * C::kKVStageBytes + (j % C::kSub) * C::kSubBytes;
        return d0 + (uint64_t)(off >> 4);
      };
      uint64_t dq[NQ];
#pragma unroll
      for (int t = 0; t < NQ; ++t)
        dq[t] = smem_desc(smem_u32(sQ + (t < C::kQTiles ? t : 0) * C::kQTileBytes), 16, 1024, kSwizzle128B);
      const uint64_t dk0 = smem_desc(smem_u32(sK), 16, 1024, kSwizzle128B);
      // V as the MN-major B operand: consecutive 64-column panels are kKVPanelBytes apart
      const uint64_t dv0 = smem_desc(smem_u32(sV), C::kKVPanelBytes, 1024, kSwizzle128B);
      bool ok = mbar_wait_warp(bar_q, 0, err, abort_flag);
      tc_fence_after();

      // S_t(j) = Q_t K_j^T into S buffer j % NS of tile t
      // g: ring position of the K / V tile (= j except with key halves)
      auto issue_s = [&](int t, int j, int g) {
        const uint64_t dk = kv_tile_desc(dk0, g, C::kStagesK);
        const uint32_t d_tmem = tmem + C::s_col(t, j % NS);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // k-step of 16 elements: 32 bytes inside a 128-byte panel, then the next panel
          const uint64_t offq = (uint64_t)(((kk >> 2) * C::kQPanelBytes + (kk & 3) * 32) >> 4);
          const uint64_t offk = (uint64_t)(((kk >> 2) * C::kKVPanelBytes + (kk & 3) * 32) >> 4);
          mma_ss_e(d_tmem, dq[t] + offq, dk + offk, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit_e(&bar_S[t * NS + j % NS]);
      };
      // O_t += P_t(j) V_j, P read from TMEM over S buffer j % NS; tile j is the
      // (j / NS)-th use of that buffer
      auto issue_pv = [&](int t, int j, int g) -> bool {
        const int buf = j % NS;
        if (!mbar_wait_warp(&bar_P[t * NS + buf], (uint32_t)(j / NS) & 1u, err, abort_flag)) return false;
        tc_fence_after();
        const uint64_t dv = kv_tile_desc(dv0, g, C::kStagesV);
        const uint32_t p_tmem = tmem + C::s_col(t, buf);
        const uint32_t d_tmem = tmem + C::o_col(t);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)  // 16 keys = 8 TMEM columns of bf16 pairs, 2048 B of V
          mma_ts_e(d_tmem, p_tmem + kk * 8, dv + (uint64_t)(kk * (2048 >> 4)), idesc_o,
                   (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_e(&bar_O[t]);
        if (j == ti[t].n_kv - 1) mma_commit_e(&bar_Fin[t]);
        return true;
      };

      if constexpr (HALVES) {
        // ring items in order (step 0, tile 0), (step 0, tile 1), (step 1, tile 0), ...:
        // S of both tiles' first items, then per step and tile P.V of the item and
        // S of the tile's next item -- the order the TMA producer loads them in
        int ik = 0, iv = 0;  // next K / V item
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (ok && ti[t].n_kv > 0) {
            ok = mbar_wait_warp(&bar_fullK[ik % C::kStagesK], (uint32_t)(ik / C::kStagesK) & 1u, err, abort_flag);
            tc_fence_after();
            if (ok) {
              issue_s(t, 0, ik);
              mma_commit_e(&bar_emptyK[ik % C::kStagesK]);
              ++ik;
            }
          }
        }
        for (int j = 0; ok && j < n_kv; ++j) {
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (ok && j < ti[t].n_kv) {
              ok = mbar_wait_warp(&bar_fullV[iv % C::kStagesV], (uint32_t)(iv / C::kStagesV) & 1u, err, abort_flag);
              tc_fence_after();
              if (ok) ok = issue_pv(t, j, iv);
              if (ok) {
                mma_commit_e(&bar_emptyV[iv % C::kStagesV]);
                ++iv;
              }
            }
            if (ok && j + 1 < ti[t].n_kv) {
              ok = mbar_wait_warp(&bar_fullK[ik % C::kStagesK], (uint32_t)(ik / C::kStagesK) & 1u, err, abort_flag);
              tc_fence_after();
              if (ok) {
                issue_s(t, j + 1, ik);
                mma_commit_e(&bar_emptyK[ik % C::kStagesK]);
                ++ik;
              }
            }
          }
        }
      } else {
      if (ok) {
        // prologue: S of the first KV tile
        ok = mbar_wait_warp(&bar_fullK[0], 0, err, abort_flag);
        tc_fence_after();
        if (ok) {
#pragma unroll
          for (int t = 0; t < NQ; ++t)
            if (ti[t].n_kv > 0) issue_s(t, 0, 0);
          if (C::kSub == 1 || n_kv == 1) mma_commit_e(&bar_emptyK[0]);
        }
      }
      // a stage is waited for at its first tile and released after its last one
      auto first_of_stage = [&](int j) { return j % C::kSub == 0; };
      auto last_of_stage = [&](int j) { return j % C::kSub == C::kSub - 1 || j == n_kv - 1; };
      for (int j = 0; ok && j < n_kv; ++j) {
        const int jn = j + 1;
        if constexpr (NS == 1) {
          // one S buffer per tile: S_t(j+1) overwrites P_t(j), so it follows P_t(j).V(j);
          // the tiles alternate so one tile's softmax runs while the other's MMAs do
          const int u = j / C::kSub, s = u % C::kStagesV;
          if (first_of_stage(j)) {
            if (!mbar_wait_warp(&bar_fullV[s], (uint32_t)(u / C::kStagesV) & 1u, err, abort_flag)) break;
            tc_fence_after();
          }
          const int un = jn / C::kSub, sn = un % C::kStagesK;
          bool k_ready = false;
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (ok && j < ti[t].n_kv) ok = issue_pv(t, j, j);
            if (ok && jn < ti[t].n_kv) {
              if (!k_ready && first_of_stage(jn)) {
                ok = mbar_wait_warp(&bar_fullK[sn], (uint32_t)(un / C::kStagesK) & 1u, err, abort_flag);
                tc_fence_after();
              }
              k_ready = true;
              if (ok) issue_s(t, jn, jn);
            }
          }
          if (!ok) break;
          if (k_ready && last_of_stage(jn)) mma_commit_e(&bar_emptyK[sn]);
          if (last_of_stage(j)) mma_commit_e(&bar_emptyV[s]);
          continue;
        }
        // S(j+1) into the other S buffer: its previous P was read by P.V(j-1), issued before
        if (jn < n_kv) {
          const int un = jn / C::kSub, sn = un % C::kStagesK;
          if (first_of_stage(jn)) {
            if (!mbar_wait_warp(&bar_fullK[sn], (uint32_t)(un / C::kStagesK) & 1u, err, abort_flag)) break;
            tc_fence_after();
          }
#pragma unroll
          for (int t = 0; t < NQ; ++t)
            if (jn < ti[t].n_kv) issue_s(t, jn, jn);
          if (last_of_stage(jn)) mma_commit_e(&bar_emptyK[sn]);
        }
        const int u = j / C::kSub, s = u % C::kStagesV;
        if (first_of_stage(j)) {
          if (!mbar_wait_warp(&bar_fullV[s], (uint32_t)(u / C::kStagesV) & 1u, err, abort_flag)) break;
          tc_fence_after();
        }
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (ok && j < ti[t].n_kv) ok = issue_pv(t, j, j);
        }
        if (!ok) break;
        if (last_of_stage(j)) mma_commit_e(&bar_emptyV[s]);
      }
      }  // HALVES
    }
  }
  } else {
    // =========================== softmax warpgroups ===========================
    if constexpr (NQ == 2) setmaxnreg_inc<C::kSoftmaxRegs>();
    const int t = warp >> 2;         // query tile of this warpgroup
    const int wq = warp & 3;         // TMEM lane quarter
    const int r = wq * 32 + lane;    // row within the tile = TMEM lane
    const TileInfo my = ti[t];
    const int qrow = my.q0 + r;       // tile row
    const int qpos = qrow / G;        // its query position
    const int qg = qrow - qpos * G;   // its head within the group
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = scale * kLog2e;
    // admissible keys of this row: [0, row_bound), and with a sliding window only
    // [row_lo, row_bound) plus the sinks [0, n_sink)
    int row_bound = khi;
    if (causal) {
      const long long rb = (long long)qpos + pos_off + 1;  // causal bound of this row
      row_bound = (int)(rb < 0 ? 0 : (rb > khi ? khi : rb));
    }
    // (32-bit, clamped: key indices are below 2^31; a bound below 0 masks nothing)
    auto clamp_key = [](long long x) { return (int)(x < -1 ? -1 : (x > 0x7FFFFFFF ? 0x7FFFFFFF : x)); };
    const int row_lo = WIN ? clamp_key((long long)qpos + pos_off - window + 1) : -1;
    // the window start of the tile's last existing row: keys below it need the mask
    const int tile_lo_max =
        WIN ? clamp_key((long long)((min(Sr, my.q0 + kPrefillTileM) - 1) / G) + pos_off - window + 1) : -1;
    float m_used = -INFINITY, l = 0.f, l_rnd = 0.f;
    bool ok = true;

    for (int j = 0; j < my.n_kv; ++j) {
      const int buf = j % NS;
      const uint32_t sph = (uint32_t)(j / NS) & 1u;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_S[t * NS + buf], sph, err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_addr = lane_addr + C::s_col(t, buf);
      uint32_t sr[BN];
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) tmem_ld32(s_addr + c0, sr + c0);
      tmem_wait_ld();
      // mask: keys at or past row_bound (causal bound or Skv), and with a window the
      // keys below the row's window that are not sinks
      const int key0 = tile_list_key(tl, HALVES ? (t == 1 ? n0 + j : j) : j) * BN;
      if (key0 + BN > my.kv_lo || (SPLIT && key0 < klo)) {
        const int lim = row_bound - key0, low = klo - key0;  // and keys below the split
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= lim || (SPLIT && c < low)) sr[c] = __float_as_uint(-INFINITY);
      }
      if (WIN && key0 < tile_lo_max && key0 + BN > n_sink) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (key0 + c < row_lo && key0 + c >= n_sink) sr[c] = __float_as_uint(-INFINITY);
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
      if (lane == 0) mbar_arrive(&bar_P[t * NS + buf]);
    }

    // ---- epilogue: O / l and LSE ----
    if (ok && my.n_kv > 0) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_Fin[t], 0, err, abort_flag))) ok = false;
      tc_fence_after();
    }
    // key halves: tile 1 hands its rows' (m, l, l_rnd) to tile 0, which merges the
    // two halves (O = f0 O_0 + f1 O_1 against the larger max) and writes the rows
    float f0 = 1.f, f1 = 0.f;
    bool have1 = false;  // warp-uniform: tile 1 held keys
    if constexpr (HALVES) {
      float* mg = reinterpret_cast<float*>(smem + C::kMergeOff) + r * 4;
      if (t == 1) {
        mg[0] = m_used;
        mg[1] = l;
        mg[2] = l_rnd;
        mg[3] = ok ? 1.f : 0.f;
        named_bar_arrive(3, 256);  // always, so tile 0 never waits for a failed tile 1
      } else {
        named_bar_sync(3, 256);
        const float m1 = mg[0], l1 = mg[1], lr1 = mg[2];
        ok = ok && mg[3] != 0.f;
        have1 = ti[1].n_kv > 0;
        if (ok && have1) {  // O_1 complete: its last P.V is done
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_Fin[1], 0, err, abort_flag))) ok = false;
          tc_fence_after();
        }
        const float m = fmaxf(m_used, m1);
        f0 = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - m);
        f1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - m);
        l = l * f0 + l1 * f1;
        l_rnd = l_rnd * f0 + lr1 * f1;
        m_used = m;
      }
    }
    if (!(HALVES && t == 1)) {
    // warp-uniform: tcgen05.ld below is a warp-collective instruction
    const bool load_o = ok && my.n_kv > 0;
    const bool have = load_o && l > 0.f;  // per row: at least one admissible key
    const float inv_l = have ? 1.f / l_rnd : 0.f;
    const bool row_ok = qrow < Sr;
    const uint32_t o_addr = lane_addr + C::o_col(t);
    const int hq = hu * G + qg;  // query head of this row
    // with key splits the row is a decode partial: part_o / part_lse [B][Hq][n_splits]
    const bool partial = SPLIT;
    const size_t prow = ((size_t)b * Hq + hq) * NSPL + sp;
    const size_t orow = partial ? prow
                                : ((size_t)ext.bq * ext.rows + ext.qbase + (size_t)(row_ok ? qpos : 0)) * Hq + hq;
    void* const out = partial ? static_cast<void*>(part_o) : o_ptr;
    // 32 columns of this row's O (merged over the key halves), or zeros
    const uint32_t o_addr1 = lane_addr + C::o_col(NQ - 1);
    auto load_o32 = [&](int c0, uint32_t* ov) {
      if (load_o) {
        tmem_ld32(o_addr + c0, ov);
        tmem_wait_ld();
        if (HALVES && have1) {
          uint32_t o1[32];
          tmem_ld32(o_addr1 + c0, o1);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            ov[e] = __float_as_uint(fmaf(__uint_as_float(ov[e]), f0, __uint_as_float(o1[e]) * f1));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0u;
      }
    };
    // (a packed varlen tile that runs past its sequence's rows would overwrite the
    // next sequence's: it keeps the per-row stores; the choice is per tile, so the
    // whole warpgroup takes the same branch)
    if (!SPLIT && o_tma && (cu_q == nullptr || my.q0 + kPrefillTileM <= Sr)) {
      // bf16 O through shared memory: every S MMA of this tile has completed (its
      // last P.V has), so the tile's Q buffer takes O in the same 128-byte-swizzled
      // layout and one TMA store per panel writes it (rows past Sq are clipped)
      uint8_t* const stile = sQ + t * C::kQTileBytes;
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
          *reinterpret_cast<uint4*>(stile + pnl * C::kQPanelBytes + r * 128 + ((cc ^ (r & 7)) << 4)) = w;
        }
      }
      fence_proxy_async_smem();
      // the warpgroup's rows are all in place (and every wait of theirs succeeded)
      const bool all_ok = bar_sync_and(1 + t, 128, ok);
      if (all_ok && my.q0 < Sr && (threadIdx.x & 127) == 0) {  // a tile past the end stores nothing
#pragma unroll
        for (int pnl = 0; pnl < C::kPanels; ++pnl)
          tma_store_5d(&tm_o, stile + pnl * C::kQPanelBytes, pnl * 64, 0, hu, ext.qbase + my.q0 / G, ext.bq);
        tma_store_commit();
        tma_store_wait_read();  // shared memory stays valid until the store has read it
      }
    } else {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        load_o32(c0, ov);
        if (row_ok && ok) {
          if (o_bf16 && !partial) {
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
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + orow * D + c0);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              dst[q4] = make_float4(__uint_as_float(ov[4 * q4 + 0]) * inv_l, __uint_as_float(ov[4 * q4 + 1]) * inv_l,
                                    __uint_as_float(ov[4 * q4 + 2]) * inv_l, __uint_as_float(ov[4 * q4 + 3]) * inv_l);
            }
          }
        }
      }
    }
    if (row_ok && ok) {
      const float lse_v = have ? (m_used + log2f(l)) * kLn2 : -INFINITY;
      if (partial) part_lse[prow] = lse_v;
      else lse_ptr[((size_t)ext.bq * Hq + hq) * ext.rows + ext.qbase + qpos] = lse_v;
    }
    }  // rows written by this warpgroup
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

// SMs of the current device
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// One launch of grid CTAs over units [unit0, ...) with configuration H.
template <int D, bool H>
cudaError_t launch_prefill_grid(const PrefillArgs& a, cudaStream_t stream, long long unit0, long long grid,
                                int row_halves) {
  using C = PrefillCfg<D, H>;
  auto kern = fmha_fwd_kernel<D, false, false, false>;
  if constexpr (H) {
    kern = a.n_splits > 1 ? fmha_fwd_kernel<D, false, true, true> : fmha_fwd_kernel<D, false, false, true>;
  } else {
    if (a.window > 0) kern = fmha_fwd_kernel<D, true, false, false>;
    else if (a.n_splits > 1) kern = fmha_fwd_kernel<D, false, true, false>;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (grid <= 0) return cudaSuccess;
  const int G = a.pack;
  const int n_splits = a.n_splits > 1 ? a.n_splits : 1;
  kern<<<(unsigned)grid, C::kThreads, C::kSmemBytes, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.o_tma, a.o, a.lse, a.Hq, a.Hkv, a.Sq, a.Skv, a.causal, a.o_bf16, a.scale,
      (a.Hq / G) * a.B, a.err, a.cu_q, a.kv_lens, a.total_q, a.window, a.n_sink, G, n_splits,
      a.split_min, a.part_o, a.part_lse, (int)unit0, row_halves);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_prefill_t(const PrefillArgs& a, cudaStream_t stream) {
  using C = PrefillCfg<D, false>;
  const int G = a.pack;
  const long long rows = (long long)a.Sq * G;
  const long long n_blocks_q = (rows + C::NQ * kPrefillTileM - 1) / (C::NQ * kPrefillTileM);
  const int n_splits = a.n_splits > 1 ? a.n_splits : 1;
  const long long units = n_blocks_q * (a.Hq / G) * a.B * n_splits;
  if (units <= 0) return cudaSuccess;
  if (2 * units > 0x7FFFFFFFLL || rows > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  if (a.halves) return launch_prefill_grid<D, true>(a, stream, 0, units, 0);
  // a causal fixed-length launch (one head per tile, no window or key splits) runs
  // on the persistent kernel, which overlaps each unit's Q load, first MMAs and O
  // epilogue with its neighbours (prefill_persist.cu)
  if (a.causal && a.window == 0 && n_splits == 1 && a.cu_q == nullptr && a.kv_lens == nullptr && G == 1)
    return launch_prefill_persistent(a, stream);
  // A non-causal fixed-length launch whose last wave is at most half full: that
  // wave's units run as two 128-row halves each, whose two query tiles take the
  // two halves of the keys (the key-halves kernel), in about half a unit's time.
  const bool plain = !a.causal && a.window == 0 && n_splits == 1 && a.cu_q == nullptr &&
                     a.kv_lens == nullptr && G == 1;
  const long long n_sm = sm_count();
  const long long tail = n_sm > 0 ? units % n_sm : 0;
  if (plain && units > n_sm && tail > 0 && 2 * tail <= n_sm) {
    cudaError_t e = launch_prefill_grid<D, false>(a, stream, 0, units - tail, 0);
    if (e != cudaSuccess) return e;
    return launch_prefill_grid<D, true>(a, stream, units - tail, 2 * tail, 1);
  }
  return launch_prefill_grid<D, false>(a, stream, 0, units, 0);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_prefill_t<64>(a, stream);
    case 128: return launch_prefill_t<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefill_empty_kv(const PrefillArgs& a, cudaStream_t stream) {
  const size_t rows = a.cu_q ? (size_t)a.total_q : (size_t)a.B * a.Sq;
  const size_t n_o = rows * a.Hq * a.d;
  const size_t n_lse = rows * a.Hq;
  if (n_o == 0) return cudaSuccess;
  fill_empty_kernel<<<1024, 256, 0, stream>>>(a.o, a.lse, n_o, n_lse, a.o_bf16);
  return cudaGetLastError();
}

}  // namespace attn
