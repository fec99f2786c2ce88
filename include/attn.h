/*
 * attn.h -- C ABI of the GB300 (sm_103a) attention-forward engine.
 *
 * Exact scaled-dot-product attention with online softmax,
 *     O = softmax(scale * Q K^T + causal mask) V,   LSE_i = ln sum_j exp(scale * q_i . k_j),
 * in two shapes: a prefill FMHA (tcgen05 tensor cores, TMEM accumulators, TMA
 * loads) and a GQA split-KV decode (per-split partials, then an LSE-weighted
 * merge) on CUDA cores.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers are DEVICE pointers owned by the caller (e.g. torch tensors'
 *    data_ptr()).  The library never frees a caller's buffer.  Per device it
 *    keeps a small word for error reporting (allocated at the first call) and,
 *    for the causal fixed-length prefill, the unit schedule of each launch
 *    shape (a few KB, uploaded at that shape's first launch, at most 256
 *    shapes; a launch that is being captured into a CUDA graph uploads nothing
 *    and takes the schedule of an earlier launch of its shape, else a simpler
 *    one).  Both are held until the process exits; a cudaDeviceReset()
 *    invalidates them: do not call the library on a device again in the same
 *    process after resetting it.
 *  - bf16 buffers hold raw bfloat16 bits (attn_bf16_t).  Every tensor is
 *    dense, row-major, contiguous in the layout stated for it, and 16-byte
 *    aligned (the TMA engine reads whole 16-byte units).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  A return of ATTN_OK means "validated and enqueued".
 *    Faults that can only be seen on the device (a pipeline wait that ran out
 *    of time) are reported by attn_sync_check().
 *  - On ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED nothing is launched and no
 *    output is written.  There is no fallback path: an unsupported shape is an
 *    error, never a slow substitute.
 *  - Empty work (B == 0, Sq == 0) is a valid no-op returning ATTN_OK.
 *
 * Causal alignment: query i of Sq sits at key position i + (Skv - Sq)
 * (bottom-right); with Sq == Skv this is the usual lower-triangular mask.  A
 * query with no admissible key (only possible when Sq > Skv) gets O = 0 and
 * LSE = -inf.  GQA: query head hq reads KV head hq / (Hq / Hkv).
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t attn_bf16_t;         /* raw bfloat16 bits */
typedef struct CUstream_st* attn_stream_t; /* == cudaStream_t */

/* status codes */
#define ATTN_OK 0
#define ATTN_ERR_INVALID_ARG (-1)    /* null/misaligned pointer, bad size, Hq % Hkv != 0, ... */
#define ATTN_ERR_UNSUPPORTED (-2)    /* head_dim not served by the entry point, unknown dtype code */
#define ATTN_ERR_CUDA (-3)           /* a CUDA runtime/driver call or a launch failed */
#define ATTN_ERR_DEVICE_TIMEOUT (-4) /* a kernel's bounded wait ran out (attn_sync_check only) */
#define ATTN_ERR_SCRATCH_TOO_SMALL (-5) /* attn_decode_noalloc: problem exceeds the static scratch */
#define ATTN_ERR_DEVICE_INPUT (-6)   /* a kernel found device-side inputs changed under it (attn_sync_check only) */

/* output dtype codes */
#define ATTN_F32 0
#define ATTN_BF16 1

/*
 * attn_prefill_fwd -- exact attention forward, prefill shape (FMHA).
 *
 * Computes, for every batch b, query head hq and query row i,
 *   O[b,i,hq,:] = sum_j P_ij V[b,j,hk,:],  P_ij = exp(S_ij - LSE_i),
 *   S_ij = scale * Q[b,i,hq,:] . K[b,j,hk,:]  (j admissible),  hk = hq / (Hq/Hkv),
 *   LSE[b,hq,i] = ln sum_j exp(S_ij)          (natural log).
 * The pages this follows: "60 . r57 -- FA KV staging double buffering
 * (REVERTED)", section 2.3 (online softmax: running row max and an
 * exp(m_old - m_new) rescale of O at every KV tile boundary, which regroups
 * the exact softmax sum); "STAGE_D.md -- FMHA Kernel Development", Kernel
 * Output (O from P = exp(S*scale - row_max), LSE from the row sum), Architecture
 * (TMA warp, MMA warp, softmax warps) and TMEM Layout (S, P and O in tensor
 * memory).  Unlike that page, O is normalised inside the kernel and LSE is in
 * natural-log units.
 *
 * Arguments
 *   q    bf16 [B][Sq][Hq][d]      queries
 *   k    bf16 [B][Skv][Hkv][d]    keys
 *   v    bf16 [B][Skv][Hkv][d]    values
 *   o    [B][Sq][Hq][d], fp32 (o_dtype = ATTN_F32) or bf16 (ATTN_BF16)
 *   lse  fp32 [B][Hq][Sq]
 *   B, Hq, Hkv, Sq, Skv   sizes: B, Sq, Skv >= 0; Hq, Hkv >= 1; Hq % Hkv == 0;
 *                         Sq, Skv < 2^31; every tensor < 2^31 rows of d elements
 *   d                     head dim: 64, 128, 256 or 512.  At 512 the fp32 O of a
 *                         128-row tile fills all of tensor memory, so O is computed
 *                         in two column halves one after the other (on CTA pairs of
 *                         256 query rows), S = Q K^T once per half (1.5x the tensor
 *                         work of the other head dims); the pages'
 *                         D1.4 of "STAGE_D.md -- FMHA Kernel Development" meets this
 *                         head dim as a shared-memory limit and splits the head
 *                         dimension, which the kernel does for Q, K, V and O.  Head
 *                         dim 512 is served by attn_prefill_fwd only (the window,
 *                         packed, variable-length and decode entry points return
 *                         ATTN_ERR_UNSUPPORTED for it)
 *   causal                0 = full attention, else bottom-right causal mask
 *   scale                 softmax scale (finite, > 0), e.g. 1/sqrt(d)
 *   o_dtype               ATTN_F32 or ATTN_BF16
 *   stream                CUDA stream the work is enqueued on
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
int attn_prefill_fwd(const attn_bf16_t* q, const attn_bf16_t* k, const attn_bf16_t* v, void* o,
                     float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                     float scale, int o_dtype, attn_stream_t stream);

/*
 * attn_prefill_window -- causal prefill over a sliding window plus attention sinks.
 *
 * As attn_prefill_fwd with causal = 1, except that query row i (key position
 * p = i + Skv - Sq) admits only the keys
 *   p - window < j <= p     (the last `window` positions, its own included)
 *   j < n_sink, j <= p      (the first n_sink positions, always visible)
 * A row with no admissible key gets O = 0 and LSE = -inf.  Only the KV tiles
 * that hold admissible keys are read: the sink tiles and the tiles of the
 * window.  This is one launch computing what "STAGE_D.md -- FMHA Kernel
 * Development", D3-D5, builds from two passes (a sliding-window branch with
 * its length and causal masks, and a sink branch) merged through their LSEs:
 * the softmax over the union of the two key sets.
 *
 * Arguments: as attn_prefill_fwd, plus
 *   window   >= 1: positions in the window (window >= Skv is plain causal attention)
 *   n_sink   >= 0: leading sink positions
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
int attn_prefill_window(const attn_bf16_t* q, const attn_bf16_t* k, const attn_bf16_t* v, void* o,
                        float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int d, int window,
                        int n_sink, float scale, int o_dtype, attn_stream_t stream);

/*
 * attn_prefill_packed -- attn_prefill_fwd with the query heads of each KV head
 * folded into the rows of the MMA tiles (head packing).
 *
 * Same arguments, layouts and results as attn_prefill_fwd (up to summation
 * order).  The G = Hq / Hkv query heads that share a KV head fill the 128 rows of
 * a query tile together: row r of a tile is position r / G, head r % G of the
 * group, so each K/V tile is streamed once per group of G heads instead of once
 * per head, and a short sequence (a decode step, a small chunk) still fills the
 * tile.  Follows "STAGE_D.md -- FMHA Kernel Development", D2 (the multi-query
 * grid: query blocks x batch, the head axis folded into the M dimension).
 * Requires d in {64, 128} and G dividing 128 (MQA: Hkv = 1, Hq <= 128 a power of
 * two); otherwise returns ATTN_ERR_UNSUPPORTED.
 */
int attn_prefill_packed(const attn_bf16_t* q, const attn_bf16_t* k, const attn_bf16_t* v, void* o,
                        float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                        float scale, int o_dtype, attn_stream_t stream);

/*
 * attn_decode_packed -- one-token decode on the tensor cores with head packing.
 *
 * For every sequence b and query head hq (hk = hq / (Hq/Hkv)):
 *   o[b,hq,:] = sum_{j < L_b} exp(s_j - lse[b,hq]) vcache[b,j,hk,:],
 *   s_j = scale * q[b,hq,:] . kcache[b,j,hk,:],   lse[b,hq] = ln sum_{j < L_b} exp(s_j),
 * L_b = kv_lens[b] -- the merged result of attn_decode_split + attn_merge, in one
 * launch and without split partials.  The G = Hq/Hkv heads of a KV head form the
 * rows of one MMA tile (the FMHA page's D2), so a decode step of G >= 8 heads per
 * KV head runs on tcgen05 instead of CUDA cores; one unit of work per (sequence,
 * KV head) streams that sequence's keys once.  Requires d in {64, 128} and
 * G <= 128 (a G that does not divide 128 leaves the tile's last 128 mod G rows
 * unused).
 *
 * Arguments
 *   q         bf16 [B][Hq][d]
 *   kcache    bf16 [B][max_kv][Hkv][d]   keys; rows >= kv_lens[b] are never admitted
 *   vcache    bf16 [B][max_kv][Hkv][d]
 *   kv_lens   int32 [B] (device)         0 <= L_b <= max_kv (clamped on the device)
 *   o         [B][Hq][d], fp32 (ATTN_F32) or bf16 (ATTN_BF16); L_b = 0 gives o = 0
 *   lse       fp32 [B][Hq]; L_b = 0 gives -inf
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
int attn_decode_packed(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                       const int* kv_lens, int B, int Hq, int Hkv, int d, int max_kv, float scale,
                       void* o, float* lse, int o_dtype, attn_stream_t stream);

/*
 * attn_decode_split_packed -- attn_decode_split on the tensor cores with head
 * packing: the same partials (part_o, part_lse), split rule, layouts and empty-split
 * convention, to be combined by attn_merge.
 *
 * Each (sequence, split, KV head) is one unit of work whose G = Hq/Hkv query
 * heads fill the rows of an MMA tile (the FMHA page's D2); splits spread a long
 * sequence's keys over several SMs ("66 . D2: explicit K+V register staging",
 * section 3.2: rows [lo, hi) of one sequence).  Requires d in {64, 128} and
 * G <= 128; part_o and part_lse 16-byte aligned.  Arguments as for
 * attn_decode_split (n_splits in [1, 1024], min_rows_per_split >= 0).
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
int attn_decode_split_packed(const attn_bf16_t* q, const attn_bf16_t* kcache,
                             const attn_bf16_t* vcache, const int* kv_lens, int B, int Hq, int Hkv,
                             int d, int max_kv, float scale, int n_splits, int min_rows_per_split,
                             float* part_o, float* part_lse, attn_stream_t stream);

/*
 * attn_prefill_varlen -- prefill of a packed batch of sequences of different
 * lengths against a KV cache (chunked prefill).
 *
 * Sequence b has Sq_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] query rows, stored
 * at rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) of q, and L_b = kv_lens[b] keys,
 * rows [0, L_b) of kcache / vcache (its earlier context followed by its own new
 * tokens).  For every such row i (0 <= i < Sq_b), query head hq (hk = hq / (Hq/Hkv)):
 *   O[cu_b + i, hq, :] = sum_j P_ij vcache[b, j, hk, :],   P_ij = exp(S_ij - LSE_i),
 *   S_ij = scale * q[cu_b + i, hq, :] . kcache[b, j, hk, :],   LSE[hq, cu_b + i] = ln sum_j exp(S_ij),
 * over the admissible keys j < L_b, and with `causal` only j <= i + (L_b - Sq_b):
 * the new rows are the last Sq_b positions of the sequence (bottom-right
 * alignment).  A row with no admissible key gets O = 0 and LSE = -inf.
 * The pages give the per-sequence key bound `kv_end` of "60 . r57 -- FA KV
 * staging double buffering (REVERTED)", section 2.2 (KV rows past the end of
 * the sequence read as zero and are never admitted); the computation per
 * sequence is the one of attn_prefill_fwd.
 *
 * Arguments
 *   q         bf16 [total_q][Hq][d]        packed queries of all sequences
 *   kcache    bf16 [B][max_kv][Hkv][d]     keys; rows >= kv_lens[b] are never admitted
 *   vcache    bf16 [B][max_kv][Hkv][d]     values
 *   o         [total_q][Hq][d], fp32 (o_dtype = ATTN_F32) or bf16 (ATTN_BF16)
 *   lse       fp32 [Hq][total_q]
 *   cu_seqlens_q  int32 [B+1] (device)     non-decreasing, cu[0] = 0, cu[B] = total_q
 *   kv_lens       int32 [B] (device)       0 <= L_b <= max_kv
 *                 (device values are trusted to be in range; they are clamped on the device)
 *   B, Hq, Hkv, total_q, max_sq, max_kv   B, total_q >= 0; Hq % Hkv == 0; max_sq >= every
 *                                          Sq_b (it sizes the grid); max_kv >= 0
 *   d, causal, scale, o_dtype, stream      as for attn_prefill_fwd
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
int attn_prefill_varlen(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                        void* o, float* lse, const int* cu_seqlens_q, const int* kv_lens, int B,
                        int Hq, int Hkv, int total_q, int max_sq, int max_kv, int d, int causal,
                        float scale, int o_dtype, attn_stream_t stream);

/*
 * attn_prefill_varlen_window -- packed variable-length prefill against a KV
 * cache with a causal sliding window and attention sinks.
 *
 * As attn_prefill_varlen with causal = 1, except that row i of sequence b (key
 * position p = i + L_b - Sq_b) admits only the keys p - window < j <= p and the
 * sinks j < n_sink (j <= p), all below L_b.  kv_lens plays the part of the
 * per-sequence window length of "STAGE_D.md -- FMHA Kernel Development", D3;
 * the window and sink sets are those of attn_prefill_window (D4, D5).
 *
 * Arguments: as attn_prefill_varlen without `causal`, plus
 *   window   >= 1: positions in the window
 *   n_sink   >= 0: leading sink positions
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
int attn_prefill_varlen_window(const attn_bf16_t* q, const attn_bf16_t* kcache,
                               const attn_bf16_t* vcache, void* o, float* lse,
                               const int* cu_seqlens_q, const int* kv_lens, int B, int Hq, int Hkv,
                               int total_q, int max_sq, int max_kv, int d, int window, int n_sink,
                               float scale, int o_dtype, attn_stream_t stream);

/*
 * attn_decode_split -- one-token GQA decode, split-KV partials.
 *
 * For every batch b, KV head hk and split s, the rows [lo, hi) of sequence b
 * (split rule below) are streamed once; the G = Hq/Hkv query heads that share
 * hk all use each loaded K/V row.  Per query head hq and split s:
 *   part_lse[b,hq,s]  = ln sum_{j in [lo,hi)} exp(s_j),   s_j = scale * q[b,hq,:] . kcache[b,j,hk,:]
 *   part_o[b,hq,s,:]  = sum_{j in [lo,hi)} exp(s_j - part_lse[b,hq,s]) vcache[b,j,hk,:]
 * i.e. each partial O is normalised within its own split (not globally), so
 * attn_merge needs only (part_o, part_lse).  An empty split (lo == hi) gets
 * part_lse = -inf and part_o = 0.
 * Split rule: chunk_b = max(ceil(L_b / n_splits), min_rows_per_split); split s
 * covers [s*chunk_b, min(L_b, (s+1)*chunk_b)).
 * Launch order (throughput only, results do not depend on it): the full splits
 * of every sequence start first, then the partial last splits by size, then
 * the empty ones.  Each CTA derives its split from kv_lens, so kv_lens must not
 * change while the call runs; a CTA that finds no split at its position (only
 * possible if it did) records ATTN_ERR_DEVICE_INPUT for attn_sync_check.
 * Follows "66 . D2: explicit K+V register staging", section 3.2 (one split =
 * rows [lo, hi) of one sequence and KV head; score, running max, running sum
 * and running O) and section 2.2 (K and V loads issued ahead of the
 * exp/shuffle chain -- here by a TMA producer warp into a shared-memory ring).
 *
 * Arguments
 *   q         bf16 [B][Hq][d]             one query token per sequence
 *   kcache    bf16 [B][max_kv][Hkv][d]    keys; rows >= kv_lens[b] are never read as data
 *   vcache    bf16 [B][max_kv][Hkv][d]    values
 *   kv_lens   int32 [B] (device)          L_b, 0 <= L_b <= max_kv (values are trusted
 *                                         to be in range; they are clamped on the device)
 *   B, Hq, Hkv, d, max_kv                 B >= 0, Hq % Hkv == 0, Hq/Hkv <= 128, d in {64,128,256},
 *                                         max_kv >= 1
 *   scale                                 softmax scale (finite, > 0)
 *   n_splits                              >= 1 and <= 1024; B * Hkv * n_splits <= 2^31 - 1
 *   min_rows_per_split                    >= 0
 *   part_o    fp32 [B][Hq][n_splits][d]   output (scratch for attn_merge)
 *   part_lse  fp32 [B][Hq][n_splits]      output
 */
int attn_decode_split(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                      const int* kv_lens, int B, int Hq, int Hkv, int d, int max_kv, float scale,
                      int n_splits, int min_rows_per_split, float* part_o, float* part_lse,
                      attn_stream_t stream);

/*
 * attn_merge -- LSE-weighted combine of split partials.
 *
 *   M = max_s part_lse[b,hq,s],  w_s = exp(part_lse[b,hq,s] - M),
 *   o[b,hq,:]  = sum_s w_s part_o[b,hq,s,:] / sum_s w_s,
 *   lse[b,hq]  = M + ln sum_s w_s.
 * Empty splits (part_lse = -inf) are skipped without reading their part_o; if
 * every split is empty, o = 0 and lse = -inf.  Follows the split-combine step
 * of "66 . D2: explicit K+V register staging", section 5.2, and the LSE merge
 * of two partial results in "STAGE_D.md -- FMHA Kernel Development", D5.
 *
 * Arguments
 *   part_o    fp32 [B][Hq][n_splits][d],  part_lse fp32 [B][Hq][n_splits]
 *   o         [B][Hq][d], fp32 or bf16 per o_dtype;  lse fp32 [B][Hq]
 *   B >= 0, Hq >= 1, n_splits in [1, 1024], d in {64, 128, 256}
 */
int attn_merge(const float* part_o, const float* part_lse, void* o, float* lse, int B, int Hq,
               int n_splits, int d, int o_dtype, attn_stream_t stream);

/*
 * attn_decode -- one-token GQA decode: the split-KV partials and their
 * LSE-weighted combine in a single launch.
 *
 * Computes what attn_decode_split followed by attn_merge computes, with the
 * same arguments, split rule and layouts, and writes the same part_o /
 * part_lse on the way; o and lse are bit-identical to those two calls.  The
 * n_splits CTAs that hold the same query heads of a sequence form a group:
 * each writes its partials, makes them visible device-wide and counts itself
 * on the group's counter, and the CTA whose count completes the group merges
 * its rows (the merge of attn_merge) and sets the counter back to zero.  This
 * is the split-combine step of "66 . D2: explicit K+V register staging",
 * section 5.2, run by the split kernel itself instead of a second launch.
 *
 * Arguments: those of attn_decode_split and of attn_merge (o, lse, o_dtype), plus
 *   counters  uint32 [B * Hq] (device, 4-byte aligned): completion counters.
 *             The caller zeroes them once; every call that completes leaves them
 *             zero, so one buffer serves any number of calls in sequence.  Calls
 *             that may run at the same time (on streams not ordered with each
 *             other) need buffers of their own.  After an error reported by
 *             attn_sync_check their contents are undefined: zero them again.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA;
 * device-side errors are reported by attn_sync_check as for attn_decode_split.
 */
int attn_decode(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                const int* kv_lens, int B, int Hq, int Hkv, int d, int max_kv, float scale,
                int n_splits, int min_rows_per_split, float* part_o, float* part_lse, void* o,
                float* lse, int o_dtype, unsigned int* counters, attn_stream_t stream);

/*
 * attn_decode_noalloc -- attn_decode_split followed by attn_merge, for callers
 * that cannot allocate device memory.  (The pages have no counterpart: this
 * entry point exists for callers, not for the method.)
 *
 * The split partials that attn_decode_split writes to a caller-provided buffer
 * live here in a fixed array of device memory owned by the library, so the
 * caller passes only inputs and outputs.  It is meant for callers that cannot
 * call cudaMalloc: code under a memory pool that has already reserved the
 * device's memory, code that must not call cudaMalloc/cudaFree because both
 * may synchronise the whole device, and plain C callers without a device
 * allocator.  Nothing is allocated per call, and no allocating library
 * routine is called.
 *
 *  - Limit: B * Hq * n_splits * (d + 1) * 4 bytes (each part rounded up to 256
 *    bytes) must fit in attn_decode_noalloc_scratch_bytes() = 24 MiB; larger
 *    problems return ATTN_ERR_SCRATCH_TOO_SMALL before any launch.  The other
 *    arguments are checked first, by the rules of attn_decode_split and
 *    attn_merge (a malformed call returns ATTN_ERR_INVALID_ARG or
 *    ATTN_ERR_UNSUPPORTED whatever its size).
 *  - The array is part of the library's device code: it is reserved on a GPU
 *    when that code is first loaded there (with CUDA's default lazy loading,
 *    at the library's first use on that device, not when the process loads
 *    the library) and stays reserved until the process exits.
 *  - The first call on a device looks up the array's device address (with that
 *    device current) and caches it; make that first call before any stream
 *    capture.  A cudaDeviceReset() invalidates that address and the library's
 *    other per-device state: do not call the library on a device again in the
 *    same process after resetting it.
 *  - All calls on a device share the array; each call writes every entry it
 *    later reads, so nothing needs to start at zero, but calls whose work
 *    overlaps on the GPU (e.g. on two streams) race on it.
 * Arguments, layouts and the split rule are those of attn_decode_split, with
 * the outputs of attn_merge: o [B][Hq][d] (fp32 or bf16 per o_dtype), lse fp32
 * [B][Hq].
 */
int attn_decode_noalloc(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                        const int* kv_lens, int B, int Hq, int Hkv, int d, int max_kv, float scale,
                        int n_splits, int min_rows_per_split, void* o, float* lse, int o_dtype,
                        attn_stream_t stream);

/* Size in bytes of the static scratch array attn_decode_noalloc uses (24 MiB). */
unsigned long long attn_decode_noalloc_scratch_bytes(void);

/*
 * attn_sync_check -- synchronise `stream`, then read and clear this device's
 * error word.  Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT (a kernel's bounded
 * wait gave up; that kernel's outputs are invalid), ATTN_ERR_DEVICE_INPUT (a
 * kernel found a device-side input inconsistent with its launch, e.g. kv_lens
 * changed while attn_decode_split ran; that call's outputs are invalid) or
 * ATTN_ERR_CUDA.  The first error recorded since the last check is reported.
 */
int attn_sync_check(attn_stream_t stream);

/* Human-readable text for a status code (static storage, never NULL). */
const char* attn_strerror(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int attn_version(void);

/*
 * attn_prefill_schedule -- the unit schedule the causal fixed-length prefill
 * runs on (host only: no GPU, no CUDA call).  (The pages have no counterpart:
 * it is how this library spreads work over SMs.)
 *
 * A unit is one 256-row query block of one (sequence, query head); the launch
 * runs one CTA per SM, each walking a list of units.  For BH = B * Hq heads, Sq
 * query rows and Skv keys on `grid` CTAs this writes offsets[grid + 1] and
 * units[n] (CTA c runs units[offsets[c] .. offsets[c+1]), in that order) and
 * returns n = ceil(Sq / 256) * BH.  Unit u is query block
 * ceil(Sq / 256) - 1 - u / BH of head u % BH.  Returns 0 (nothing written) when
 * the launch deals its units in waves instead (more than 64 units per CTA);
 * ATTN_ERR_INVALID_ARG for bad arguments or max_units < n.
 */
int attn_prefill_schedule(int BH, int Sq, int Skv, int causal, int grid, int* offsets, int* units,
                          int max_units);

/*
 * attn_debug_wait_timeout -- test hook for the bounded-wait machinery.
 * Launches one CTA that waits on an mbarrier nobody arrives on, with a limit of
 * `limit_ns` nanoseconds (1e3 .. 1e10), then records ATTN_ERR_DEVICE_TIMEOUT in
 * the error word and exits.  attn_sync_check() then reports the timeout.  The
 * kernel never hangs and never faults.
 */
int attn_debug_wait_timeout(unsigned long long limit_ns, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
