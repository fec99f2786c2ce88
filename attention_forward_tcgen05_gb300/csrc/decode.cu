// decode.cu -- one-token GQA decode on CUDA cores: split-KV partials and the
// LSE-weighted merge.
//
// What one split computes follows "66 . D2: explicit K+V register staging",
// section 3.2: for the rows [lo, hi) of one sequence and one KV head, every
// query head of the GQA group takes the score s = (q . k) * scale, keeps a
// running max, a running sum and a running O, and rescales both by
// exp(m_old - m_new) when the max grows.  Section 2.2 of that page moves the
// K and V loads ahead of the exp/shuffle dependency chain; here the same idea
// is carried by the GB300 copy engine: producer warps issue TMA loads (64 rows
// of K and of V per stage) into a shared-memory ring, so the loads of later
// stages are in flight while the consumer warps work on earlier ones.  The
// copy engine's throughput is set by the number of boxes far more than by
// their size (about one box per 300 cycles per SM up to 16 KB), so a stage is
// one 64-row box per 128-byte panel: 32-row boxes capped the kernel at about
// 14 bytes per cycle per SM, below the HBM rate.
//
// Work mapping: one CTA per split unit (batch, KV head, split), 6 warps; a
// launch with few units spreads each group's query heads over several CTAs.
// Consumer warps 0..3 form two pairs; pair p owns ring stage p and takes the
// stages u = p, p+2, p+4, ... of the unit, warp h of the pair the rows
// [32h, 32h+32) of each, for all G query heads of the group, so every loaded
// K/V row serves all G heads.  Warp 4 streams K and warp 5 streams V with
// TMA; a pair hands its K half back right after the score phase, so its next
// K stage loads during softmax and P.V.
// Per tile: scores with lane = row (the head dim of that row from shared
// memory against q, kept in shared memory as bf16: every lane reads all of q
// for every row, and shared-memory wavefronts, not HBM, were the limit with
// an fp32 copy), scaled by scale * log2(e) once per score, warp-shuffle max,
// exp2 on the MUFU, then P.V with lane = d/32 dims and each row's weights
// broadcast from shared memory (a shuffle per row and head instead was about
// 1.5x slower).  The score products take q and k as bf16 straight from shared
// memory into a mixed-precision fma (bf16 x bf16 + fp32, exact products, one
// rounding per step, the same result as fp32 fmas of the widened values); the
// bf16 -> fp32 conversions this removes were most of the score loop's
// instructions (0.73 -> 0.83 of the copy bandwidth on a ragged 64-sequence
// batch).  P.V runs on packed fp32 pairs (fma.f32x2).  At the end the four warps' partial
// (m, l, O) are merged through shared memory and the split's normalised O
// and LSE are written.  Everything is fp32 on CUDA cores; no tensor cores.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kConsumerWarps = 4;                   // one ring stage each
constexpr int kDecodeThreads = (kConsumerWarps + 2) * 32;  // + K producer + V producer

template <int D, int GMAX>
struct DecodeCfg {
  static constexpr int kTile = 32;                     // rows per consumer warp and stage
  static constexpr int kStageRows = kDecodeStageRows;  // rows per stage (one TMA box per panel)
  static constexpr int kWarpsPerStage = kStageRows / kTile;
  static constexpr int kStages = kConsumerWarps / kWarpsPerStage;
  static constexpr int kPanels = D / 64;               // 128-byte swizzled panels per row
  static constexpr int kPanelBytes = kStageRows * 128; // one panel of one stage
  static constexpr int kKBytes = kPanels * kPanelBytes;  // the K half of a stage (V half: same)
  static constexpr int kStageBytes = 2 * kKBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static_assert(kConsumerWarps % kWarpsPerStage == 0, "whole warp groups per stage");
  static constexpr int kQBytes = GMAX * D * 2;                             // bf16 q [GMAX][D]
  static constexpr int kPBytes = kConsumerWarps * kTile * GMAX * 4;        // p [warp][row][g]
  static constexpr int kBarOffset = kRingBytes + kQBytes + kPBytes;
  static constexpr int kBarBytes = 4 * kStages * 8 + 16;  // fullK, fullV, emptyK, emptyV, abort
  static constexpr int kSmemBytes = kBarOffset + kBarBytes + 1024;  // + align slack
  // three CTAs per SM for small head groups, two otherwise (register budget)
  static constexpr int kMinBlocks = GMAX <= 4 ? 3 : 2;
};

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }
// two bf16 (low, high half of x) as an fp32 pair
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t x) { return f2pack(bf16lo(x), bf16hi(x)); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return v;
}

// ---- launch order of the split units ----
// Unit (b, s) holds clamp(L_b - s*chunk_b, 0, chunk_b) rows.  CTAs start in index
// order and an SM takes the next one when a slot frees, so a ragged batch ends
// soonest when the long units start first and the short ones fill the end (the
// longest-first list-scheduling rule).  Every unit of a sequence but its last
// non-empty one is full, so the order is: all full units, then the partial last
// units by size (kOrderBuckets buckets of chunk / kOrderBuckets rows, largest
// first, batch order within a bucket), then the empty units.  Each CTA derives
// its unit from kv_lens with two warp-wide passes over the batch.  Batches above
// kOrderMaxBatch take the batch-major order instead (the passes would cost more
// than the tail they save).
constexpr int kOrderBuckets = 16;
constexpr int kOrderMaxBatch = 1024;

struct SplitShape {
  int nf;  // full units (chunk rows each)
  int hp;  // 1 if a partial unit follows them
  int bk;  // size bucket of the partial unit, or -1
  int ne;  // empty units
};

// the split rule of the kernel: chunk = max(ceil(L / n_splits), min_rows, 1)
__device__ __forceinline__ SplitShape split_shape(int L, int max_kv, int n_splits, int min_rows) {
  L = L < 0 ? 0 : (L > max_kv ? max_kv : L);
  int chunk = L / n_splits + (L % n_splits != 0 ? 1 : 0);
  chunk = max(max(chunk, min_rows), 1);
  SplitShape r;
  r.nf = L / chunk;
  const int rem = L - r.nf * chunk;
  r.hp = rem > 0 ? 1 : 0;
  r.bk = r.hp ? (int)((long long)rem * kOrderBuckets / chunk) : -1;
  r.ne = n_splits - r.nf - r.hp;
  return r;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int x = __shfl_up_sync(0xFFFFFFFFu, v, off);
    if (lane >= off) v += x;
  }
  return v;
}

// (b, s) of the unit at position p of the launch order, for every lane of the
// calling warp; (-1, -1) if p is past the last unit.
__device__ __noinline__ int2 unit_at(int p, const int* __restrict__ kv_lens, int B, int max_kv, int n_splits,
                                      int min_rows, int lane) {
  auto shape_of = [&](int b) {
    return b < B ? split_shape(kv_lens[b], max_kv, n_splits, min_rows) : SplitShape{0, 0, -1, 0};
  };
  int F = 0, P = 0;  // full and partial units of the batch
  for (int b0 = 0; b0 < B; b0 += 32) {
    const SplitShape sh = shape_of(b0 + lane);
    F += (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)sh.nf);
    P += __popc(__ballot_sync(0xFFFFFFFFu, sh.hp != 0));
  }
  if (p < F || p >= F + P) {
    // a full unit (the p-th, batch-major) or an empty one (the (p-F-P)-th)
    const bool full = p < F;
    const int q = full ? p : p - F - P;
    int carry = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const SplitShape sh = shape_of(b0 + lane);
      const int n = full ? sh.nf : sh.ne;
      const int incl = warp_incl_scan(n, lane) + carry, excl = incl - n;
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, excl <= q && q < incl);
      if (hit) {
        const int src = __ffs(hit) - 1;
        const int first = full ? 0 : sh.nf + sh.hp;  // first unit of the class in the sequence
        const int s = __shfl_sync(0xFFFFFFFFu, first + q - excl, src);
        return make_int2(b0 + src, s);
      }
      carry = __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    return make_int2(-1, -1);
  }
  // a partial unit: count the buckets (lane k < kOrderBuckets holds bucket k)
  int cnt = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const SplitShape sh = shape_of(b0 + lane);
#pragma unroll
    for (int k = 0; k < kOrderBuckets; ++k) {
      const int c = __popc(__ballot_sync(0xFFFFFFFFu, sh.bk == k));
      if (lane == k) cnt += c;
    }
  }
  int j = p - F, K = -1;
  for (int k = kOrderBuckets - 1; k >= 0; --k) {  // largest bucket first
    const int c = __shfl_sync(0xFFFFFFFFu, cnt, k);
    if (j < c) {
      K = k;
      break;
    }
    j -= c;
  }
  if (K < 0) return make_int2(-1, -1);
  for (int b0 = 0; b0 < B; b0 += 32) {  // the j-th sequence of bucket K, in batch order
    const SplitShape sh = shape_of(b0 + lane);
    const unsigned m = __ballot_sync(0xFFFFFFFFu, sh.bk == K);
    const int c = __popc(m);
    if (j < c) {
      const unsigned below = (1u << lane) - 1u;
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, ((m >> lane) & 1u) && __popc(m & below) == j);
      const int src = __ffs(hit) - 1;
      return make_int2(b0 + src, __shfl_sync(0xFFFFFFFFu, sh.nf, src));
    }
    j -= c;
  }
  return make_int2(-1, -1);
}

__device__ __forceinline__ void consumer_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Non-empty splits whose partial rows a merge warp loads at once: eight covers
// the common split counts in one round trip (four took two on eight splits).
constexpr int kMergeBatch = 8;

// The LSE-weighted combine of the n_splits partials of one (sequence, query
// head) row, by one warp: lane = DPL consecutive dims.  The partials are read
// through L2 (ld.global.cg): in the fused decode other CTAs of the same launch
// wrote them, and this SM's L1 may not see those writes.
template <int D>
__device__ __noinline__ void merge_row(const float* __restrict__ part_o,
                                          const float* __restrict__ part_lse, void* o,
                                          float* __restrict__ lse, size_t row, int n_splits,
                                          int o_bf16, int lane) {
  constexpr int DPL = D / 32;
  const float* pl = part_lse + row * n_splits;
  const float* po = part_o + row * n_splits * D + lane * DPL;
  float M = -INFINITY;
  for (int s = lane; s < n_splits; s += 32) M = fmaxf(M, __ldcg(pl + s));
  M = warp_max(M);
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < n_splits; s0 += 32) {
      // lane j holds the weight of split s0 + j (0 for empty or missing splits)
      const int s = s0 + lane;
      const float ls = s < n_splits ? __ldcg(pl + s) : -INFINITY;
      const float w = ls == -INFINITY ? 0.f : ex2_approx((ls - M) * kLog2e);
      wsum += w;
      uint32_t live = __ballot_sync(0xFFFFFFFFu, w > 0.f);  // empty splits are never read
      while (live) {
        // up to kMergeBatch non-empty splits per round: their loads are issued together
        int idx[kMergeBatch];
        float wk[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          idx[u] = live ? __ffs(live) - 1 : -1;
          if (live) live &= live - 1;
          wk[u] = __shfl_sync(0xFFFFFFFFu, w, idx[u] < 0 ? 0 : idx[u]);
        }
        float x[kMergeBatch][DPL];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          if (idx[u] >= 0) {
            const float* src = po + (size_t)(s0 + idx[u]) * D;
#pragma unroll
            for (int e = 0; e < DPL; e += 2) {
              const float2 v2 = __ldcg(reinterpret_cast<const float2*>(src + e));
              x[u][e] = v2.x;
              x[u][e + 1] = v2.y;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          if (idx[u] >= 0) {
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wk[u], x[u][e], acc[e]);
          }
        }
      }
    }
    wsum = warp_sum(wsum);
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  if (o_bf16) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(o) + row * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; e += 2) {
      *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    }
  } else {
    float* dst = reinterpret_cast<float*>(o) + row * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; e += 2) {
      *reinterpret_cast<float2*>(dst + e) = make_float2(acc[e] * inv, acc[e + 1] * inv);
    }
  }
  if (lane == 0) lse[row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

// The combine fused into the split launch ("66 . D2: explicit K+V register
// staging", section 5.2, without a launch of its own).  The n_splits CTAs that
// hold the same query heads of a sequence form a group with one completion
// counter, indexed by the group's first (sequence, query head) row.  Each CTA,
// once its partials are written, fences them and counts
// itself; the CTA that takes the count to n_splits merges the group's rows
// into o and lse and puts the counter back to zero, so the counters are zero
// again when the launch ends.  Called by the first NWARPS warps of the CTA
// together; `sync` is their barrier.
template <int D, int NWARPS, class Sync>
__device__ __forceinline__ void combine_if_last(unsigned* done, int n_splits,
                                                const float* part_o, const float* part_lse,
                                                void* o, float* lse, size_t row0, int G,
                                                int o_bf16, Sync sync) {
  __shared__ int last_sh;
  __threadfence();  // this thread's partials are visible device-wide before the count
  sync();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(done, 1u);
    const int last = prev + 1u == (unsigned)n_splits;
    if (last) {
      __threadfence();      // the other CTAs' partials are read after their counts
      atomicExch(done, 0u);  // ready for the next launch
    }
    last_sh = last;
  }
  sync();
  if (!last_sh) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int g = warp; g < G; g += NWARPS)
    merge_row<D>(part_o, part_lse, o, lse, row0 + g, n_splits, o_bf16, lane);
}

// One CTA per split unit (batch b, KV head hk, split s).  Consumer warp w owns
// ring stage w and takes tiles w, w+4, w+8, ... of the unit, for all G query
// heads of the group.  A stage has a K half and a V half with their own
// barriers: the warp hands the K half back as soon as its scores are done, so
// the K producer warp refills it with the warp's next K tile while the warp is
// still in softmax and P.V; the V producer warp refills the V half after P.V.
template <int D, int GMAX, bool SPLIT_HEADS>
__global__ void __launch_bounds__(kDecodeThreads, DecodeCfg<D, GMAX>::kMinBlocks)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const uint16_t* __restrict__ q,
                        const int* __restrict__ kv_lens, float* __restrict__ part_o,
                        float* __restrict__ part_lse, int Hq, int Hkv, int max_kv, int n_splits,
                        int min_rows, float scale, int heads_per_cta, int ordered, int B,
                        uint32_t* err, unsigned* __restrict__ done, void* o,
                        float* __restrict__ lse, int o_bf16) {
  using C = DecodeCfg<D, GMAX>;
  constexpr int DPL = D / 32;   // output dims per lane in the P.V phase
  constexpr int DP2 = DPL / 2;  // ... as fp32 pairs
  // CTA = (unit, KV head, head group): the query heads [g0, g0 + G) of the KV
  // head's group (all of them unless a small launch splits the group across
  // CTAs, which then re-read the same K/V rows from L2).  The CTAs of one unit
  // are adjacent, so the KV heads of the same rows are read together.
  const int Gall = Hq / Hkv;
  const int n_hg = SPLIT_HEADS ? (Gall + heads_per_cta - 1) / heads_per_cta : 1;
  const int per_unit = Hkv * n_hg;
  const int pos = (int)(blockIdx.x / per_unit), w_in = (int)(blockIdx.x % per_unit);
  const int hk = w_in / n_hg;
  int g0 = 0, G = Gall;
  if constexpr (SPLIT_HEADS) {
    g0 = (w_in % n_hg) * heads_per_cta;
    G = min(heads_per_cta, Gall - g0);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int b, s_idx;
  if (ordered) {
    __shared__ int2 unit_sh;
    if (warp == 0) {
      const int2 u = unit_at(pos, kv_lens, B, max_kv, n_splits, min_rows, lane);
      if (lane == 0) unit_sh = u;
    }
    __syncthreads();
    b = unit_sh.x;
    s_idx = unit_sh.y;
    if (b < 0) {
      // Only reachable if kv_lens changed while the launch ran (the launch order is
      // derived from it by every CTA): this unit's partials are not written, so the
      // call is reported as failed through the error word rather than leaving stale
      // partials for the merge to combine silently.
      if (threadIdx.x == 0) atomicCAS(err, kErrNone, kErrBadShape);
      return;
    }
  } else {
    b = pos / n_splits;
    s_idx = pos % n_splits;
  }

  // ---- split bounds: chunk = max(ceil(L / n_splits), min_rows) ----
  int L = kv_lens[b];
  L = L < 0 ? 0 : (L > max_kv ? max_kv : L);
  long long chunk = ((long long)L + n_splits - 1) / n_splits;
  if (chunk < min_rows) chunk = min_rows;
  if (chunk < 1) chunk = 1;
  const long long lo_ll = (long long)s_idx * chunk, hi_ll = lo_ll + chunk;
  const int lo = (int)(lo_ll < L ? lo_ll : L), hi = (int)(hi_ll < L ? hi_ll : L);
  const size_t row_base = ((size_t)b * Hq + (size_t)hk * Gall + g0) * n_splits + s_idx;  // head g: + g*n_splits

  if (lo >= hi) {  // empty split: o = 0, lse = -inf; nothing is read
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
      const int g = i / D, t = i % D;
      part_o[(row_base + (size_t)g * n_splits) * D + t] = 0.f;
      if (t == 0) part_lse[row_base + (size_t)g * n_splits] = -INFINITY;
    }
    if (done) {
      const size_t orow0 = (size_t)b * Hq + (size_t)hk * Gall + g0;
      combine_if_last<D, kDecodeThreads / 32>(done + orow0, n_splits, part_o, part_lse, o, lse, orow0,
                                              G, o_bf16, [] { __syncthreads(); });
    }
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;                                                          // [warp] K|V
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem + C::kRingBytes);  // [GMAX][D] bf16
  uint64_t* fullK = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* fullV = fullK + C::kStages;
  uint64_t* emptyK = fullV + C::kStages;
  uint64_t* emptyV = emptyK + C::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(emptyV + C::kStages);

  const int U = (hi - lo + C::kStageRows - 1) / C::kStageRows;  // stages in this split

  if (threadIdx.x == 0) {
    for (int w = 0; w < C::kStages; ++w) {
      mbar_init(&fullK[w], 1);
      mbar_init(&fullV[w], 1);
      mbar_init(&emptyK[w], C::kWarpsPerStage);  // every warp of the stage's group releases it
      mbar_init(&emptyV[w], C::kWarpsPerStage);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // q of the group, bf16 as given; scores are scaled into the log2 domain later
  const float qscale = scale * kLog2e;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int g = i / D, t = i % D;
    qs[g * D + t] = q[((size_t)b * Hq + (size_t)hk * Gall + g0 + g) * D + t];
  }
  for (int i = threadIdx.x; i < (GMAX - G) * D; i += blockDim.x) qs[G * D + i] = 0;
  __syncthreads();

  if (warp >= kConsumerWarps) {
    // ================= producer warps: warp 4 streams K, warp 5 streams V =================
    // Stage u of the unit goes to ring slot u % kStages (its (u / kStages)-th
    // use).  The whole warp runs the loop; one elected lane issues each copy.
    const bool is_k = warp == kConsumerWarps;
    const CUtensorMap* map = is_k ? &tm_k : &tm_v;
    uint64_t* fullX = is_k ? fullK : fullV;
    uint64_t* emptyX = is_k ? emptyK : emptyV;
    if (lane == 0) tma_prefetch_desc(map);
    const uint64_t pol = l2_policy_evict_first();
    int u = 0;
    for (; u < U; ++u) {
      const int w = u % C::kStages, k = u / C::kStages;
      if (!mbar_wait_warp(&emptyX[w], (k & 1) ^ 1, err, abort_flag)) break;
      mbar_arrive_expect_tx_e(&fullX[w], C::kKBytes);
      uint8_t* dst = ring + w * C::kStageBytes + (is_k ? 0 : C::kKBytes);
      const int row = lo + u * C::kStageRows;
#pragma unroll
      for (int p = 0; p < C::kPanels; ++p)
        tma_load_4d_hint_e(dst + p * C::kPanelBytes, map, &fullX[w], p * 64, hk, row, b, pol);
    }
    if (u < U && lane == 0) {
      // aborted: let the copies already issued land before the CTA exits
      for (int v = (u - C::kStages > 0 ? u - C::kStages : 0); v < u; ++v)
        mbar_wait(&fullX[v % C::kStages], (v / C::kStages) & 1, nullptr, nullptr, 100000000ull);
    }
    return;  // the producers take no part in the combine
  }

  // ================= consumer warps =================
  float m[GMAX], lsum[GMAX];
  uint64_t o2[GMAX][DP2];  // O as fp32 pairs: dims lane*DPL + 2e, +1
#pragma unroll
  for (int g = 0; g < GMAX; ++g) {
    m[g] = -INFINITY;
    lsum[g] = 0.f;
#pragma unroll
    for (int e = 0; e < DP2; ++e) o2[g][e] = f2pack(0.f, 0.f);
  }
  float* pw = reinterpret_cast<float*>(smem + C::kRingBytes + C::kQBytes) + warp * C::kTile * GMAX;
  const int slot = warp / C::kWarpsPerStage;    // ring slot of this warp's group
  const int half = warp % C::kWarpsPerStage;    // its 32 rows within each stage
  // this warp's rows of a stage: rows [32*half, 32*half + 32) of every panel
  const uint8_t* kt = ring + slot * C::kStageBytes + half * C::kTile * 128;
  const uint8_t* vt = kt + C::kKBytes;

  bool ok = true;
  for (int i = 0, u = slot; u < U; ++i, u += C::kStages) {
    const uint32_t par = (uint32_t)i & 1u;
    const int row0 = lo + u * C::kStageRows + half * C::kTile;
    // rows of this warp in the stage: 0 for the upper half of a short last stage,
    // which the warp still waits for and releases (the stage's barriers count it)
    const int nrows = max(0, min(C::kTile, hi - row0));
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&fullK[slot], par, err, abort_flag))) {
      ok = false;
      break;
    }
    if (nrows == 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&emptyK[slot]);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&fullV[slot], par, err, abort_flag))) {
        ok = false;
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&emptyV[slot]);
      continue;
    }

    // ---- scores: lane = row; fp32 pairs along the head dim ----
    float acl[GMAX], ach[GMAX];
#pragma unroll
    for (int g = 0; g < GMAX; ++g) acl[g] = ach[g] = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const int p = c >> 3, cc = c & 7;
      const uint4 kv = *reinterpret_cast<const uint4*>(kt + p * C::kPanelBytes + lane * 128 +
                                                       ((cc ^ (lane & 7)) << 4));
#pragma unroll
      for (int g = 0; g < GMAX; ++g) {
        if (g < G) {
          const uint4 qv = *reinterpret_cast<const uint4*>(qs + g * D + c * 8);  // 8 bf16, broadcast
          fma_bf16x2_f32(qv.x, kv.x, acl[g], ach[g]);
          fma_bf16x2_f32(qv.y, kv.y, acl[g], ach[g]);
          fma_bf16x2_f32(qv.z, kv.z, acl[g], ach[g]);
          fma_bf16x2_f32(qv.w, kv.w, acl[g], ach[g]);
        }
      }
    }
    // the K half of the stage is no longer needed by this warp: once both warps of
    // the group are done the K producer may refill it
    __syncwarp();
    if (lane == 0) mbar_arrive(&emptyK[slot]);
    const bool valid = lane < nrows;

    // ---- online softmax per query head (log2 domain) ----
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
      if (g < G) {
        const float sv = valid ? (acl[g] + ach[g]) * qscale : -INFINITY;
        const float tmax = warp_max(sv);  // finite: every tile has >= 1 valid row
        const float m_new = fmaxf(m[g], tmax);
        const float corr = ex2_approx(m[g] - m_new);  // m = -inf -> 0
        const float pv = ex2_approx(sv - m_new);      // invalid -> 0
        lsum[g] = fmaf(lsum[g], corr, pv);           // per-lane partial sum
        m[g] = m_new;
        const uint64_t c2 = f2pack(corr, corr);
#pragma unroll
        for (int e = 0; e < DP2; ++e) o2[g][e] = mul2(o2[g][e], c2);
        pw[lane * GMAX + g] = pv;
      }
    }
    __syncwarp();
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&fullV[slot], par, err, abort_flag))) {
      ok = false;
      break;
    }

    // ---- O += P V: lane = DPL consecutive dims ----
#pragma unroll 2
    for (int r = 0; r < nrows; ++r) {
      uint64_t vf[DP2];
      if constexpr (D == 64) {
        const uint32_t x = *reinterpret_cast<const uint32_t*>(
            vt + r * 128 + (((lane >> 2) ^ (r & 7)) << 4) + (lane & 3) * 4);
        vf[0] = bf16x2_to_f2(x);
      } else if constexpr (D == 128) {
        const uint2 x = *reinterpret_cast<const uint2*>(
            vt + (lane >> 4) * C::kPanelBytes + r * 128 + ((((lane & 15) >> 1) ^ (r & 7)) << 4) +
            (lane & 1) * 8);
        vf[0] = bf16x2_to_f2(x.x);
        vf[1] = bf16x2_to_f2(x.y);
      } else {
        const uint4 x = *reinterpret_cast<const uint4*>(vt + (lane >> 3) * C::kPanelBytes + r * 128 +
                                                        (((lane & 7) ^ (r & 7)) << 4));
        vf[0] = bf16x2_to_f2(x.x);
        vf[1] = bf16x2_to_f2(x.y);
        vf[2] = bf16x2_to_f2(x.z);
        vf[3] = bf16x2_to_f2(x.w);
      }
      const float* pr = pw + r * GMAX;
#pragma unroll
      for (int g4 = 0; g4 < GMAX; g4 += 4) {
        if (g4 < G) {
          const float4 p4 = *reinterpret_cast<const float4*>(pr + g4);
          const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            const uint64_t p2 = f2pack(pp[gg], pp[gg]);
#pragma unroll
            for (int e = 0; e < DP2; ++e) o2[g4 + gg][e] = fma2(p2, vf[e], o2[g4 + gg][e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&emptyV[slot]);
  }

  // ---- combine the consumer warps' partials through shared memory ----
  consumer_bar_sync();  // every consumer is done with its stage
  float* comb = reinterpret_cast<float*>(ring);  // [warp][g][D + 2]: o[0..D), m, l
  static_assert(kConsumerWarps * GMAX * (D + 2) * 4 <= C::kRingBytes, "combine area");
#pragma unroll
  for (int g = 0; g < GMAX; ++g) {
    if (g < G) {
      const float lw = warp_sum(lsum[g]);
      float* cw = comb + (warp * GMAX + g) * (D + 2);
#pragma unroll
      for (int e = 0; e < DP2; ++e) f2unpack(o2[g][e], cw[lane * DPL + 2 * e], cw[lane * DPL + 2 * e + 1]);
      if (lane == 0) {
        cw[D] = m[g];
        cw[D + 1] = lw;
      }
    }
  }
  // the four warps agree on whether every wait of the CTA succeeded
  const bool good = bar_sync_and(1, kConsumerWarps * 32, ok && *abort_flag == 0);
  if (good) {
    for (int idx = threadIdx.x; idx < G * D; idx += kConsumerWarps * 32) {
      const int g = idx / D, t = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, comb[(w * GMAX + g) * (D + 2) + D]);
      float Lsum = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float* cw = comb + (w * GMAX + g) * (D + 2);
        const float f = ex2_approx(cw[D] - M);  // warps without tiles: m = -inf -> 0
        Lsum = fmaf(cw[D + 1], f, Lsum);
        acc = fmaf(cw[t], f, acc);
      }
      const size_t row = row_base + (size_t)g * n_splits;
      part_o[row * D + t] = acc / Lsum;
      if (t == 0) part_lse[row] = (M + log2f(Lsum)) * kLn2;
    }
  }
  if (done) {  // counted even after a timeout (which the error word reports), so the count stays whole
    const size_t orow0 = (row_base - s_idx) / n_splits;  // (sequence, first query head) row
    combine_if_last<D, kConsumerWarps>(done + orow0, n_splits, part_o, part_lse, o, lse, orow0, G,
                                       o_bf16, [] { consumer_bar_sync(); });
  }
}

template <int D>
__global__ void __launch_bounds__(128)
    merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, void* o,
                 float* __restrict__ lse, int rows, int n_splits, int o_bf16) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  merge_row<D>(part_o, part_lse, o, lse, (size_t)row, n_splits, o_bf16, threadIdx.x & 31);
}

template <int D, int GMAX, bool SPLIT_HEADS>
cudaError_t launch_decode_t(const DecodeArgs& a, int heads_per_cta, cudaStream_t stream) {
  using C = DecodeCfg<D, GMAX>;
  auto kern = decode_split_kernel<D, GMAX, SPLIT_HEADS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int G = a.Hq / a.Hkv;
  const int n_hg = SPLIT_HEADS ? (G + heads_per_cta - 1) / heads_per_cta : 1;
  const long long ctas = (long long)a.B * a.n_splits * a.Hkv * n_hg;
  if (ctas > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const int ordered = a.B <= kOrderMaxBatch ? 1 : 0;
  kern<<<(unsigned)ctas, kDecodeThreads, C::kSmemBytes, stream>>>(
      a.tm_k, a.tm_v, a.q, a.kv_lens, a.part_o, a.part_lse, a.Hq, a.Hkv, a.max_kv, a.n_splits,
      a.min_rows, a.scale, heads_per_cta, ordered, a.B, a.err, a.done, a.o, a.lse, a.o_bf16);
  return cudaGetLastError();
}

// Query heads per CTA.  A launch with fewer than kSmallUnits (batch, KV head,
// split) units is latency-bound (one sequence of 1641 keys in 8 splits is 32
// CTAs on 152 SMs), so its head groups are spread over more CTAs.  A CTA holds
// at most kMaxHeadsPerCta heads (the register budget of the consumer warps);
// larger groups are always spread, their CTAs reading the same K/V rows (the
// CTAs of one unit are adjacent, so the re-reads are L2 hits).
constexpr int kSmallUnits = 128;

template <int D>
cudaError_t launch_decode_g(const DecodeArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  const long long units = (long long)a.B * a.Hkv * a.n_splits;
  int hpc = G;
  if (units < kSmallUnits && G > 1) {
    const int want = (int)((kSmallUnits + units - 1) / units);  // head groups wanted
    const int n_hg = want < G ? want : G;
    hpc = (G + n_hg - 1) / n_hg;
  }
  if (hpc > kMaxHeadsPerCta) {
    const int n_hg = (G + kMaxHeadsPerCta - 1) / kMaxHeadsPerCta;
    hpc = (G + n_hg - 1) / n_hg;
  }
  if (hpc < G) {
    if (hpc <= 4) return launch_decode_t<D, 4, true>(a, hpc, stream);
    if (hpc <= 8) return launch_decode_t<D, 8, true>(a, hpc, stream);
    return launch_decode_t<D, 16, true>(a, hpc, stream);
  }
  if (hpc <= 4) return launch_decode_t<D, 4, false>(a, hpc, stream);
  if (hpc <= 8) return launch_decode_t<D, 8, false>(a, hpc, stream);
  return launch_decode_t<D, 16, false>(a, hpc, stream);
}

}  // namespace

cudaError_t launch_decode_split(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_decode_g<64>(a, stream);
    case 128: return launch_decode_g<128>(a, stream);
    case 256: return launch_decode_g<256>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int rows = a.B * a.Hq;
  const dim3 grid((rows + 3) / 4);
  switch (a.d) {
    case 64:
      merge_kernel<64><<<grid, 128, 0, stream>>>(a.part_o, a.part_lse, a.o, a.lse, rows, a.n_splits, a.o_bf16);
      break;
    case 128:
      merge_kernel<128><<<grid, 128, 0, stream>>>(a.part_o, a.part_lse, a.o, a.lse, rows, a.n_splits, a.o_bf16);
      break;
    case 256:
      merge_kernel<256><<<grid, 128, 0, stream>>>(a.part_o, a.part_lse, a.o, a.lse, rows, a.n_splits, a.o_bf16);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace attn
