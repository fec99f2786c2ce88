// internal.h -- launch interface between the C-ABI layer (attn_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <vector>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Prefill launch description (already validated by the C-ABI layer).
// Fixed-length batches: cu_q == nullptr, q/o [B][Sq][Hq][d], k/v [B][Skv][Hkv][d],
// lse [B][Hq][Sq]; with kv_lens != nullptr sequence b has only the keys
// [0, kv_lens[b]) (its Sq queries are its last positions).  Packed
// variable-length batches (cu_q != nullptr): sequence b has rows
// [cu_q[b], cu_q[b+1]) of q/o [total_q][Hq][d] and lse [Hq][total_q]; its keys are
// rows [0, kv_lens[b]) of k/v [B][Skv][Hkv][d] (Skv = the cache's max_kv); Sq is
// the longest sequence (it sizes the grid).
// Head packing (pack = G > 1, single-CTA kernel only): the G query heads of one KV
// head fill the rows of a query tile, row r = position r / G, head r % G of the
// group, so a tile holds 128 / G positions.
struct PrefillArgs {
  CUtensorMap tm_o;              // bf16 O of the single-CTA kernel when o_tma: the Q map's shape
  int o_tma;                     // 1: O leaves through shared memory and TMA stores
  CUtensorMap tm_q, tm_k, tm_v;  // K, V (and Q of the pair kernel): 4-D maps {d, H, S, B},
                                 // box {64, 1, rows, 1}, 128B swizzle: rows = kPrefillTileM
                                 // for Q, prefill_k_box_rows(d) for K, kPrefillKVStageRows
                                 // for V.  Q of the single-CTA kernel: 5-D map
                                 // {d, G, Hq/G, S, B}, box {64, G, 1, 128/G, 1}.
  void* o;                       // [B][Sq][Hq][d], fp32 or bf16
  float* lse;                    // [B][Hq][Sq]
  int B, Hq, Hkv, Sq, Skv, d, causal, o_bf16;
  float scale;
  uint32_t* err;                 // device error word
  const int* cu_q;               // [B+1] packed query offsets, or nullptr
  const int* kv_lens;            // [B] keys per sequence (varlen only)
  int total_q;                   // rows of the packed q (varlen only)
  int window;                    // > 0: causal sliding window of this many positions
  int n_sink;                    // with a window: the first n_sink keys stay admissible
  int pack;                      // query rows per position (G); 1 = one head per tile
  // key splits (one-token decode with kv_lens, single-CTA kernel): n_splits > 1
  // writes per-split partials part_o [B][Hq][n_splits][d] (fp32, normalised within
  // the split) and part_lse [B][Hq][n_splits] instead of o / lse; split s of a
  // sequence with L keys covers [s*chunk, min(L, (s+1)*chunk)),
  // chunk = max(ceil(L / n_splits), split_min)
  int n_splits, split_min;
  // one query position per sequence with its G <= 128 rows in the first query tile:
  // the second tile takes the second half of the keys (merged in the epilogue)
  int halves;
  float* part_o;
  float* part_lse;
};

#ifdef __CUDACC__
// Extent of sequence b inside one prefill launch (see PrefillArgs).
struct SeqExtent {
  int Sq, Skv;     // query rows and keys of this sequence
  int qbase;       // first row of this sequence in q / o / lse
  int bq;          // batch coordinate of the q map and of the o / lse slabs
  long long rows;  // rows per batch slab of o / lse
};
__device__ __forceinline__ SeqExtent seq_extent(int b, int Sq, int Skv, const int* cu_q,
                                                const int* kv_lens, int total_q) {
  SeqExtent e;
  if (cu_q == nullptr) {
    e.Sq = Sq; e.Skv = Skv; e.qbase = 0; e.bq = b; e.rows = Sq;
    if (kv_lens != nullptr) {  // fixed queries, per-sequence keys (decode)
      const int kl = kv_lens[b];
      e.Skv = kl < 0 ? 0 : (kl > Skv ? Skv : kl);
    }
    return e;
  }
  // offsets and lengths are clamped to the buffers the caller described
  int c0 = cu_q[b], c1 = cu_q[b + 1];
  c0 = c0 < 0 ? 0 : (c0 > total_q ? total_q : c0);
  c1 = c1 < c0 ? c0 : (c1 > total_q ? total_q : c1);
  int kl = kv_lens[b];
  kl = kl < 0 ? 0 : (kl > Skv ? Skv : kl);
  e.Sq = min(c1 - c0, Sq); e.Skv = kl; e.qbase = c0; e.bq = 0; e.rows = total_q;
  return e;
}

// KV tiles a CTA visits with a sliding window: the sink tiles, then the tiles
// from the window start of the CTA's first query row up to its causal bound;
// the tiles in between hold no admissible key for any of its rows.  List entry
// u holds key tile u for u < gap_at and key tile u + gap after that.
struct TileList {
  int gap_at, gap;
};
__device__ __forceinline__ TileList tile_list(long long first_row_pos, int n_kv, int window,
                                              int n_sink, int Skv, int BN) {
  TileList L;
  L.gap_at = n_kv;
  L.gap = 0;
  if (window <= 0 || n_kv <= 0) return L;
  const int sink_keys = n_sink < Skv ? n_sink : Skv;
  int sink_tiles = (sink_keys + BN - 1) / BN;
  if (sink_tiles > n_kv) sink_tiles = n_kv;
  const long long lo = first_row_pos - window + 1;  // first key of the first row's window
  const int w0 = lo <= 0 ? 0 : (int)(lo / BN < n_kv ? lo / BN : n_kv);
  if (w0 > sink_tiles) {
    L.gap_at = sink_tiles;
    L.gap = w0 - sink_tiles;
  }
  return L;
}
// list entries holding the key tiles [0, n_key_tiles)
__device__ __forceinline__ int tile_list_len(const TileList& L, int n_key_tiles) {
  return n_key_tiles <= L.gap_at ? n_key_tiles : (n_key_tiles - L.gap > L.gap_at ? n_key_tiles - L.gap : L.gap_at);
}
__device__ __forceinline__ int tile_list_key(const TileList& L, int u) { return u < L.gap_at ? u : u + L.gap; }
#endif

// Decode-split launch description.
struct DecodeArgs {
  CUtensorMap tm_k, tm_v;  // 4-D maps {d, Hkv, max_kv, B}, box {64, 1, kDecodeStageRows, 1}, 128B swizzle
  const uint16_t* q;       // [B][Hq][d] bf16
  const int* kv_lens;      // [B]
  float* part_o;           // [B][Hq][n_splits][d]
  float* part_lse;         // [B][Hq][n_splits]
  int B, Hq, Hkv, d, max_kv, n_splits, min_rows;
  float scale;
  uint32_t* err;
  // fused combine (all null for partials only): completion counters [B * Hq],
  // one per group at its first (sequence, query head) row, zero on entry and
  // zero again on exit; and the merged outputs
  unsigned* done;
  void* o;       // [B][Hq][d], fp32 or bf16 (o_bf16)
  float* lse;    // [B][Hq]
  int o_bf16;
};

struct MergeArgs {
  const float* part_o;
  const float* part_lse;
  void* o;
  float* lse;
  int B, Hq, n_splits, d, o_bf16;
};

// Rows of a K / V stage loaded by one TMA box in the decode kernel (two
// consumer warps share a stage, 32 rows each).
constexpr int kDecodeStageRows = 64;
// Query heads one decode CTA computes; a larger GQA group is spread over
// ceil(G / kMaxHeadsPerCta) CTAs.  kMaxDecodeGroup bounds G = Hq / Hkv.
constexpr int kMaxHeadsPerCta = 16;
constexpr int kMaxDecodeGroup = 128;
// Rows of a Q tile in the prefill kernel, and of one TMA-loaded K / V stage
// (the kernel may compute on sub-tiles of a stage).
constexpr int kPrefillTileM = 128;
constexpr int kPrefillKVStageRows = 128;
// Head dims served by the CTA-pair kernel (prefill_pair.cu); there each CTA
// loads 64 of the 128 K rows of a tile, so the K map's box is 64 rows high.
// d = 256 runs faster on pairs (1.6 PFLOP/s against 1.24 on the head-dim
// sweep); d = 128 runs faster on single CTAs with two query tiles.
constexpr bool prefill_uses_pair(int d) { return d == 256; }
constexpr int prefill_k_box_rows(int d) { return prefill_uses_pair(d) ? kPrefillKVStageRows / 2 : kPrefillKVStageRows; }

// Host-side argument rules of attn_decode_split and attn_merge (ATTN_OK, or the
// status the entry point returns).  check_parts / check_partials = false skips the
// partial buffers (part_o, part_lse), which attn_decode_noalloc supplies itself.
int check_decode_split_args(const void* q, const void* kcache, const void* vcache, const int* kv_lens,
                            int B, int Hq, int Hkv, int d, int max_kv, float scale, int n_splits,
                            int min_rows, const void* part_o, const void* part_lse, bool check_parts);
int check_merge_args(const void* part_o, const void* part_lse, const void* o, const void* lse, int B,
                     int Hq, int n_splits, int d, int o_dtype, bool check_partials);

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_pair(const PrefillArgs& a, cudaStream_t stream);
// Persistent single-CTA kernel (prefill_persist.cu): fixed-length batches, one head
// per tile (pack = 1), no window, key splits or kv_lens; d in {64, 128}.
cudaError_t launch_prefill_persistent(const PrefillArgs& a, cudaStream_t stream);
// Head dimension 512 (prefill_d512.cu): fixed-length batches, causal or not; O in
// two column halves (S recomputed for the second), on CTA pairs of 256 query rows.
// Maps: Q 4-D with 128-row boxes, K boxes of 64 rows, V boxes of
// kD512PairVBoxRows rows.
cudaError_t launch_prefill_d512(const PrefillArgs& a, cudaStream_t stream);
// The CTA-pair kernel's ring: kD512PairRingBytes of shared memory in slots of
// kD512PairSlotBytes (three of 32 KB: measured against six of 16 KB and twelve of
// 8 KB, every ring item costs a cross-SM round trip, so fewer, larger items win);
// a V panel of an item holds kD512PairVBoxRows keys (the V map's box height).
constexpr int kD512PairRingBytes = 6 * 16384;
constexpr int kD512PairSlotBytes = 32768;
constexpr int kD512PairVBoxRows = kD512PairSlotBytes >= 16384 ? 128 : kD512PairSlotBytes / 128;
cudaError_t launch_prefill_empty_kv(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_decode_split(const DecodeArgs& a, cudaStream_t stream);
// The persistent prefill's unit schedule for BH = B * Hq heads over `grid` CTAs:
// sched = offsets[grid + 1] followed by each CTA's units; returns the unit count,
// 0 when the launch keeps the wave deal (sched left empty), -1 on bad arguments.
int build_prefill_schedule(int BH, int Sq, int Skv, int causal, int grid, std::vector<int>& sched);
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(uint64_t limit_ns, uint32_t* err, cudaStream_t stream);

}  // namespace attn
