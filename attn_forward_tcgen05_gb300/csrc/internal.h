// internal.h -- launch interface between the C-ABI layer (attn_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Prefill launch description (already validated by the C-ABI layer).
struct PrefillArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 4-D maps {d, H, S, B}, box {64, 1, rows, 1}, 128B swizzle:
                                 // rows = kPrefillTileM for Q, prefill_k_box_rows(d) for K,
                                 // kPrefillKVStageRows for V
  void* o;                       // [B][Sq][Hq][d], fp32 or bf16
  float* lse;                    // [B][Hq][Sq]
  int B, Hq, Hkv, Sq, Skv, d, causal, o_bf16;
  float scale;
  uint32_t* err;                 // device error word
};

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
// Rows of a Q tile in the prefill kernel, and of one TMA-loaded K / V stage
// (the kernel may compute on sub-tiles of a stage).
constexpr int kPrefillTileM = 128;
constexpr int kPrefillKVStageRows = 128;
// Head dims served by the CTA-pair kernel (prefill_pair.cu); there each CTA
// loads 64 of the 128 K rows of a tile, so the K map's box is 64 rows high.
// d = 256 runs faster on pairs (1.6 PFLOP/s against 1.24 on the head-dim
// sweep); d = 128 runs faster on single CTAs with two query tiles, so its pair
// instantiation is built only when ATTN_PREFILL_PAIR_D128 is defined to 1.
#ifndef ATTN_PREFILL_PAIR_D128
#define ATTN_PREFILL_PAIR_D128 0
#endif
constexpr bool prefill_uses_pair(int d) { return d == 256 || (ATTN_PREFILL_PAIR_D128 && d == 128); }
constexpr int prefill_k_box_rows(int d) { return prefill_uses_pair(d) ? kPrefillKVStageRows / 2 : kPrefillKVStageRows; }

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_pair(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_empty_kv(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_decode_split(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(uint64_t limit_ns, uint32_t* err, cudaStream_t stream);

}  // namespace attn
