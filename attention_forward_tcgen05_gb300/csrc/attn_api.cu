// attn_api.cu -- the C ABI declared in include/attn.h: argument validation,
// TMA tensor-map encoding, kernel launches and device error reporting.
//
// The library keeps one static device word per device (g_attn_err) for
// errors that only the device can see (a bounded pipeline wait that ran out).
// Its device address is looked up once per device with cudaGetSymbolAddress
// and handed to every kernel; attn_sync_check() reads and clears it.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "attn.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

__device__ uint32_t g_attn_err;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_err_ptr[kMaxDevices] = {nullptr};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device(int* dev) { return cudaGetDevice(dev) == cudaSuccess ? 0 : -1; }

// Device address of this device's error word (looked up once per device).
uint32_t* err_word() {
  int dev = 0;
  if (current_device(&dev) != 0 || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_err) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_err_ptr[dev];
}

EncodeTiledFn encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

// 4-D bf16 tensor map over a [n3][n2][n1][n0] row-major tensor (n0 innermost),
// box {64, 1, box_rows, 1}, 128-byte swizzle, zero fill out of bounds.
int encode_bf16_4d(CUtensorMap* map, const void* base, uint64_t n0, uint64_t n1, uint64_t n2,
                   uint64_t n3, uint32_t box_rows) {
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return ATTN_ERR_CUDA;
  const cuuint64_t dims[4] = {n0, n1, n2, n3};
  const cuuint64_t strides[3] = {n0 * 2, n0 * n1 * 2, n0 * n1 * n2 * 2};
  const cuuint32_t box[4] = {64, 1, box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 5-D bf16 tensor map for the query tiles of the single-CTA prefill kernel over a
// [nb][ns][Hq][d] row-major tensor, viewed as {d, G, Hq/G, ns, nb}: box
// {64, G, 1, 128/G, 1} holds 128/G positions x the G heads of one group, 128
// rows of 128 bytes in shared memory (row = position-in-box * G + head-in-group).
int encode_bf16_q5d(CUtensorMap* map, const void* base, uint64_t d, uint64_t G, uint64_t Hq,
                    uint64_t ns, uint64_t nb) {
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return ATTN_ERR_CUDA;
  const cuuint64_t dims[5] = {d, G, Hq / G, ns, nb};
  const cuuint64_t strides[4] = {d * 2, d * G * 2, d * Hq * 2, d * Hq * ns * 2};
  const cuuint32_t box[5] = {64, (cuuint32_t)G, 1, (cuuint32_t)(attn::kPrefillTileM / G), 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_dim(int d) { return d == 64 || d == 128 || d == 256; }
// head dims of the fixed-length prefill (attn_prefill_fwd): also 512
bool ok_dim_prefill(int d) { return ok_dim(d) || d == 512; }
bool ok_scale(float s) { return std::isfinite(s) && s > 0.f; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace

namespace attn {

int check_decode_split_args(const void* q, const void* kcache, const void* vcache, const int* kv_lens,
                            int B, int Hq, int Hkv, int d, int max_kv, float scale, int n_splits,
                            int min_rows, const void* part_o, const void* part_lse, bool check_parts) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq / Hkv > kMaxDecodeGroup || max_kv < 1)
    return ATTN_ERR_INVALID_ARG;
  if (n_splits < 1 || n_splits > 1024 || min_rows < 0 || !ok_scale(scale)) return ATTN_ERR_INVALID_ARG;
  // one CTA per (sequence, KV head, split, head group) in a 1-D grid: groups above
  // kMaxHeadsPerCta heads take several CTAs (launches of fewer than 128 units
  // also spread head groups, and stay far below the limit)
  const long long n_hg = (Hq / Hkv + kMaxHeadsPerCta - 1) / kMaxHeadsPerCta;
  if ((long long)B * Hkv * n_splits * n_hg > 0x7FFFFFFFLL) return ATTN_ERR_INVALID_ARG;
  if (!ok_dim(d)) return ATTN_ERR_UNSUPPORTED;
  if (B == 0) return ATTN_OK;
  if (!q || !kcache || !vcache || !kv_lens) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || (reinterpret_cast<uintptr_t>(kv_lens) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (check_parts && (!part_o || !part_lse || !aligned16(part_o) ||
                      (reinterpret_cast<uintptr_t>(part_lse) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if ((long long)B * max_kv * Hkv >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

int check_merge_args(const void* part_o, const void* part_lse, const void* o, const void* lse, int B,
                     int Hq, int n_splits, int d, int o_dtype, bool check_partials) {
  if (B < 0 || Hq < 1 || n_splits < 1 || n_splits > 1024) return ATTN_ERR_INVALID_ARG;
  if (!ok_dim(d) || (o_dtype != ATTN_F32 && o_dtype != ATTN_BF16)) return ATTN_ERR_UNSUPPORTED;
  if (B == 0) return ATTN_OK;
  if (!o || !lse || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (check_partials && (!part_o || !part_lse || !aligned16(part_o) ||
                         (reinterpret_cast<uintptr_t>(part_lse) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if ((long long)B * Hq >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

}  // namespace attn

// kv_lens (optional): keys per sequence, each sequence's Sq queries being its last
// positions; pack: query heads folded into the tile rows (single-CTA kernel only).
static int prefill_impl(const attn_bf16_t* q, const attn_bf16_t* k, const attn_bf16_t* v, void* o,
                        float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                        int window, int n_sink, float scale, int o_dtype, attn_stream_t stream,
                        const int* kv_lens = nullptr, int pack = 1, int n_splits = 1,
                        int split_min = 0, float* part_o = nullptr, float* part_lse = nullptr) {
  if (B < 0 || Sq < 0 || Skv < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!ok_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (!ok_dim_prefill(d) || (o_dtype != ATTN_F32 && o_dtype != ATTN_BF16)) return ATTN_ERR_UNSUPPORTED;
  // head dim 512: plain fixed-length prefill only (no window, packing, key splits or kv_lens)
  const bool d512 = d == 512;
  if (d512 && (window != 0 || pack != 1 || n_splits > 1 || kv_lens != nullptr)) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Sq == 0) return ATTN_OK;
  if (!q || !o || !lse || !aligned16(q) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  if (Skv > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return ATTN_ERR_INVALID_ARG;
  // row counts of every tensor must fit the kernels' 32-bit row indices
  if ((long long)B * Sq * Hq >= (1LL << 31) || (long long)B * Skv * Hkv >= (1LL << 31))
    return ATTN_ERR_INVALID_ARG;
  attn::PrefillArgs a;
  std::memset(&a, 0, sizeof(a));
  a.o = o;
  a.lse = lse;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.Sq = Sq; a.Skv = Skv; a.d = d;
  a.causal = causal ? 1 : 0;
  a.o_bf16 = o_dtype == ATTN_BF16 ? 1 : 0;
  a.scale = scale;
  a.window = window;
  a.n_sink = n_sink;
  a.kv_lens = kv_lens;
  a.pack = pack;
  a.n_splits = n_splits;
  a.split_min = split_min;
  // a one-token decode (one position, kv_lens): its head rows fill one query tile,
  // so the second tile takes the second half of each sequence's (or key split's) keys
  a.halves = (kv_lens != nullptr && Sq == 1 && window == 0 &&
              (long long)pack <= attn::kPrefillTileM && !attn::prefill_uses_pair(d)) ? 1 : 0;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.err = err_word();
  if (a.err == nullptr) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (Skv == 0) return from_cuda(attn::launch_prefill_empty_kv(a, s));
  if (d512) {
    int rc = encode_bf16_4d(&a.tm_q, q, d, Hq, Sq, B, attn::kPrefillTileM);
    if (rc == ATTN_OK) rc = encode_bf16_4d(&a.tm_k, k, d, Hkv, Skv, B, attn::kPrefillKVStageRows / 2);
    if (rc == ATTN_OK) rc = encode_bf16_4d(&a.tm_v, v, d, Hkv, Skv, B, attn::kD512PairVBoxRows);
    if (rc != ATTN_OK) return rc;
    return from_cuda(attn::launch_prefill_d512(a, s));
  }
  const bool pair = attn::prefill_uses_pair(d);
  if (pair && pack != 1) return ATTN_ERR_UNSUPPORTED;
  int rc = pair ? encode_bf16_4d(&a.tm_q, q, d, Hq, Sq, B, attn::kPrefillTileM)
                : encode_bf16_q5d(&a.tm_q, q, d, pack, Hq, Sq, B);
  // bf16 O of the single-CTA kernel leaves through TMA stores (same shape as Q)
  a.o_tma = (!pair && o_dtype == ATTN_BF16 && n_splits <= 1) ? 1 : 0;
  if (rc == ATTN_OK && a.o_tma) rc = encode_bf16_q5d(&a.tm_o, o, d, pack, Hq, Sq, B);
  if (rc == ATTN_OK) rc = encode_bf16_4d(&a.tm_k, k, d, Hkv, Skv, B, attn::prefill_k_box_rows(d));
  if (rc == ATTN_OK) rc = encode_bf16_4d(&a.tm_v, v, d, Hkv, Skv, B, attn::kPrefillKVStageRows);
  if (rc != ATTN_OK) return rc;
  return from_cuda(pair ? attn::launch_prefill_pair(a, s) : attn::launch_prefill(a, s));
}

static int varlen_impl(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                       void* o, float* lse, const int* cu_seqlens_q, const int* kv_lens, int B, int Hq,
                       int Hkv, int total_q, int max_sq, int max_kv, int d, int causal, int window,
                       int n_sink, float scale, int o_dtype, attn_stream_t stream) {
  if (B < 0 || total_q < 0 || max_sq < 0 || max_kv < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!ok_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (!ok_dim(d) || (o_dtype != ATTN_F32 && o_dtype != ATTN_BF16)) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || total_q == 0 || max_sq == 0) return ATTN_OK;
  if (!q || !o || !lse || !aligned16(q) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_INVALID_ARG;
  if (!cu_seqlens_q || !kv_lens || (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3) ||
      (reinterpret_cast<uintptr_t>(kv_lens) & 3))
    return ATTN_ERR_INVALID_ARG;
  if (max_kv > 0 && (!kcache || !vcache || !aligned16(kcache) || !aligned16(vcache)))
    return ATTN_ERR_INVALID_ARG;
  if ((long long)total_q * Hq >= (1LL << 31) || (long long)B * max_kv * Hkv >= (1LL << 31))
    return ATTN_ERR_INVALID_ARG;
  attn::PrefillArgs a;
  std::memset(&a, 0, sizeof(a));
  a.o = o;
  a.lse = lse;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.Sq = max_sq; a.Skv = max_kv; a.d = d;
  a.causal = causal ? 1 : 0;
  a.o_bf16 = o_dtype == ATTN_BF16 ? 1 : 0;
  a.scale = scale;
  a.window = window;
  a.n_sink = n_sink;
  a.cu_q = cu_seqlens_q;
  a.kv_lens = kv_lens;
  a.pack = 1;
  a.total_q = total_q;
  a.err = err_word();
  if (a.err == nullptr) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (max_kv == 0) return from_cuda(attn::launch_prefill_empty_kv(a, s));
  // packed q is one batch slab of total_q rows; the cache keeps its batch dimension
  const bool pair = attn::prefill_uses_pair(d);
  int rc = pair ? encode_bf16_4d(&a.tm_q, q, d, Hq, total_q, 1, attn::kPrefillTileM)
                : encode_bf16_q5d(&a.tm_q, q, d, 1, Hq, total_q, 1);
  if (rc == ATTN_OK) rc = encode_bf16_4d(&a.tm_k, kcache, d, Hkv, max_kv, B, attn::prefill_k_box_rows(d));
  if (rc == ATTN_OK) rc = encode_bf16_4d(&a.tm_v, vcache, d, Hkv, max_kv, B, attn::kPrefillKVStageRows);
  // bf16 O of whole tiles leaves through TMA stores (the kernel keeps per-row stores
  // for a sequence's last, partial tile)
  a.o_tma = (!pair && o_dtype == ATTN_BF16) ? 1 : 0;
  if (rc == ATTN_OK && a.o_tma) rc = encode_bf16_q5d(&a.tm_o, o, d, 1, Hq, total_q, 1);
  if (rc != ATTN_OK) return rc;
  return from_cuda(pair ? attn::launch_prefill_pair(a, s) : attn::launch_prefill(a, s));
}

extern "C" {

int attn_version(void) { return 10000; }

const char* attn_strerror(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer, bad size or head ratio)";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration (head dim or dtype code)";
    case ATTN_ERR_CUDA: return "CUDA runtime or launch error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel's bounded pipeline wait timed out";
    case ATTN_ERR_SCRATCH_TOO_SMALL: return "problem too large for the library's static decode scratch (24 MiB)";
    case ATTN_ERR_DEVICE_INPUT: return "a kernel found a device-side input (kv_lens) changed while it ran";
    default: return "unknown status";
  }
}

int attn_prefill_fwd(const attn_bf16_t* q, const attn_bf16_t* k, const attn_bf16_t* v, void* o,
                     float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                     float scale, int o_dtype, attn_stream_t stream) {
  return prefill_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, causal, 0, 0, scale, o_dtype, stream);
}

int attn_prefill_window(const attn_bf16_t* q, const attn_bf16_t* k, const attn_bf16_t* v, void* o,
                        float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int d, int window,
                        int n_sink, float scale, int o_dtype, attn_stream_t stream) {
  if (window < 1 || n_sink < 0) return ATTN_ERR_INVALID_ARG;
  return prefill_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, 1, window, n_sink, scale, o_dtype, stream);
}

// head packing needs the single-CTA kernel and at most 128 head rows per group; a
// prefill also needs the group to tile the 128 rows (so that tiles hold whole
// positions), a one-token decode (one position, in the first tile) does not
static bool packable(int Hq, int Hkv, int d, bool one_position = false) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return false;
  const int G = Hq / Hkv;
  return (d == 64 || d == 128) && !attn::prefill_uses_pair(d) && G <= attn::kPrefillTileM &&
         (one_position || attn::kPrefillTileM % G == 0);
}

int attn_prefill_packed(const attn_bf16_t* q, const attn_bf16_t* k, const attn_bf16_t* v, void* o,
                        float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                        float scale, int o_dtype, attn_stream_t stream) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!packable(Hq, Hkv, d)) return ATTN_ERR_UNSUPPORTED;
  return prefill_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, causal, 0, 0, scale, o_dtype, stream,
                      nullptr, Hq / Hkv);
}

int attn_decode_packed(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                       const int* kv_lens, int B, int Hq, int Hkv, int d, int max_kv, float scale,
                       void* o, float* lse, int o_dtype, attn_stream_t stream) {
  if (B < 0 || max_kv < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!ok_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (!packable(Hq, Hkv, d, true) || (o_dtype != ATTN_F32 && o_dtype != ATTN_BF16)) return ATTN_ERR_UNSUPPORTED;
  if (B == 0) return ATTN_OK;
  if (!kv_lens || (reinterpret_cast<uintptr_t>(kv_lens) & 3)) return ATTN_ERR_INVALID_ARG;
  // one query position per sequence, the last one: causal admits keys [0, kv_lens[b])
  return prefill_impl(q, kcache, vcache, o, lse, B, Hq, Hkv, 1, max_kv, d, 1, 0, 0, scale, o_dtype,
                      stream, kv_lens, Hq / Hkv);
}

int attn_decode_split_packed(const attn_bf16_t* q, const attn_bf16_t* kcache,
                             const attn_bf16_t* vcache, const int* kv_lens, int B, int Hq, int Hkv,
                             int d, int max_kv, float scale, int n_splits, int min_rows_per_split,
                             float* part_o, float* part_lse, attn_stream_t stream) {
  if (B < 0 || max_kv < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (n_splits < 1 || n_splits > 1024 || min_rows_per_split < 0 || !ok_scale(scale))
    return ATTN_ERR_INVALID_ARG;
  if (!packable(Hq, Hkv, d, true)) return ATTN_ERR_UNSUPPORTED;
  if (B == 0) return ATTN_OK;
  if (!kv_lens || (reinterpret_cast<uintptr_t>(kv_lens) & 3)) return ATTN_ERR_INVALID_ARG;
  if (!part_o || !part_lse || !aligned16(part_o) || !aligned16(part_lse)) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * Hq * n_splits >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
  if (max_kv == 0) {
    // no keys anywhere: every partial is empty (o = 0, lse = -inf)
    return prefill_impl(q, kcache, vcache, part_o, part_lse, B * n_splits, Hq, Hkv, 1, 0, d, 1, 0, 0,
                        scale, ATTN_F32, stream);
  }
  return prefill_impl(q, kcache, vcache, part_o, part_lse, B, Hq, Hkv, 1, max_kv, d, 1, 0, 0, scale,
                      ATTN_F32, stream, kv_lens, Hq / Hkv, n_splits, min_rows_per_split, part_o,
                      part_lse);
}

int attn_prefill_varlen(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                        void* o, float* lse, const int* cu_seqlens_q, const int* kv_lens, int B,
                        int Hq, int Hkv, int total_q, int max_sq, int max_kv, int d, int causal,
                        float scale, int o_dtype, attn_stream_t stream) {
  return varlen_impl(q, kcache, vcache, o, lse, cu_seqlens_q, kv_lens, B, Hq, Hkv, total_q, max_sq,
                     max_kv, d, causal, 0, 0, scale, o_dtype, stream);
}

int attn_prefill_varlen_window(const attn_bf16_t* q, const attn_bf16_t* kcache,
                               const attn_bf16_t* vcache, void* o, float* lse,
                               const int* cu_seqlens_q, const int* kv_lens, int B, int Hq, int Hkv,
                               int total_q, int max_sq, int max_kv, int d, int window, int n_sink,
                               float scale, int o_dtype, attn_stream_t stream) {
  if (window < 1 || n_sink < 0) return ATTN_ERR_INVALID_ARG;
  return varlen_impl(q, kcache, vcache, o, lse, cu_seqlens_q, kv_lens, B, Hq, Hkv, total_q, max_sq,
                     max_kv, d, 1, window, n_sink, scale, o_dtype, stream);
}

// split partials, and with `done` set their combine into (o, lse) in the same launch
static int decode_launch(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                         const int* kv_lens, int B, int Hq, int Hkv, int d, int max_kv, float scale,
                         int n_splits, int min_rows_per_split, float* part_o, float* part_lse,
                         unsigned* done, void* o, float* lse, int o_dtype, attn_stream_t stream) {
  attn::DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q; a.kv_lens = kv_lens; a.part_o = part_o; a.part_lse = part_lse;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.max_kv = max_kv;
  a.n_splits = n_splits; a.min_rows = min_rows_per_split; a.scale = scale;
  a.done = done; a.o = o; a.lse = lse; a.o_bf16 = o_dtype == ATTN_BF16 ? 1 : 0;
  a.err = err_word();
  if (a.err == nullptr) return ATTN_ERR_CUDA;
  int rc = encode_bf16_4d(&a.tm_k, kcache, d, Hkv, max_kv, B, attn::kDecodeStageRows);
  if (rc == ATTN_OK) rc = encode_bf16_4d(&a.tm_v, vcache, d, Hkv, max_kv, B, attn::kDecodeStageRows);
  if (rc != ATTN_OK) return rc;
  return from_cuda(attn::launch_decode_split(a, reinterpret_cast<cudaStream_t>(stream)));
}

int attn_decode_split(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                      const int* kv_lens, int B, int Hq, int Hkv, int d, int max_kv, float scale,
                      int n_splits, int min_rows_per_split, float* part_o, float* part_lse,
                      attn_stream_t stream) {
  const int rc0 = attn::check_decode_split_args(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale,
                                                n_splits, min_rows_per_split, part_o, part_lse, true);
  if (rc0 != ATTN_OK || B == 0) return rc0;
  return decode_launch(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale, n_splits,
                       min_rows_per_split, part_o, part_lse, nullptr, nullptr, nullptr, ATTN_F32, stream);
}

int attn_decode(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                const int* kv_lens, int B, int Hq, int Hkv, int d, int max_kv, float scale,
                int n_splits, int min_rows_per_split, float* part_o, float* part_lse, void* o,
                float* lse, int o_dtype, unsigned int* counters, attn_stream_t stream) {
  int rc = attn::check_decode_split_args(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale,
                                         n_splits, min_rows_per_split, part_o, part_lse, true);
  if (rc == ATTN_OK) rc = attn::check_merge_args(part_o, part_lse, o, lse, B, Hq, n_splits, d, o_dtype, true);
  if (rc != ATTN_OK || B == 0) return rc;
  if (!counters || (reinterpret_cast<uintptr_t>(counters) & 3u)) return ATTN_ERR_INVALID_ARG;
  return decode_launch(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale, n_splits,
                       min_rows_per_split, part_o, part_lse, counters, o, lse, o_dtype, stream);
}

int attn_merge(const float* part_o, const float* part_lse, void* o, float* lse, int B, int Hq,
               int n_splits, int d, int o_dtype, attn_stream_t stream) {
  const int rc0 = attn::check_merge_args(part_o, part_lse, o, lse, B, Hq, n_splits, d, o_dtype, true);
  if (rc0 != ATTN_OK || B == 0) return rc0;
  attn::MergeArgs a;
  a.part_o = part_o; a.part_lse = part_lse; a.o = o; a.lse = lse;
  a.B = B; a.Hq = Hq; a.n_splits = n_splits; a.d = d; a.o_bf16 = o_dtype == ATTN_BF16 ? 1 : 0;
  return from_cuda(attn::launch_merge(a, reinterpret_cast<cudaStream_t>(stream)));
}

int attn_sync_check(attn_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  uint32_t* e = err_word();
  if (e == nullptr) return ATTN_ERR_CUDA;
  uint32_t h = 0;
  if (cudaMemcpy(&h, e, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (h != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(e, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
    return h == attn::kErrBadShape ? ATTN_ERR_DEVICE_INPUT : ATTN_ERR_DEVICE_TIMEOUT;
  }
  return ATTN_OK;
}

int attn_prefill_schedule(int BH, int Sq, int Skv, int causal, int grid, int* offsets, int* units,
                          int max_units) {
  if (BH < 1 || Sq < 0 || Skv < 0 || grid < 1 || max_units < 0 || !offsets || (max_units > 0 && !units))
    return ATTN_ERR_INVALID_ARG;
  std::vector<int> sched;
  const int n = attn::build_prefill_schedule(BH, Sq, Skv, causal ? 1 : 0, grid, sched);
  if (n < 0) return ATTN_ERR_INVALID_ARG;
  if (n == 0) return 0;
  if (n > max_units) return ATTN_ERR_INVALID_ARG;
  std::memcpy(offsets, sched.data(), sizeof(int) * ((size_t)grid + 1));
  std::memcpy(units, sched.data() + grid + 1, sizeof(int) * (size_t)n);
  return n;
}

int attn_debug_wait_timeout(unsigned long long limit_ns, attn_stream_t stream) {
  if (limit_ns < 1000ull || limit_ns > 10000000000ull) return ATTN_ERR_INVALID_ARG;
  uint32_t* e = err_word();
  if (e == nullptr) return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_wait_timeout_probe(limit_ns, e, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace attn {
namespace {
// One CTA waits on an mbarrier that nothing ever arrives on; the bounded wait
// gives up after limit_ns, records the timeout and the kernel returns.
__global__ void wait_timeout_probe_kernel(uint64_t limit_ns, uint32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, err, &abort_flag, limit_ns);
}
}  // namespace

cudaError_t launch_wait_timeout_probe(uint64_t limit_ns, uint32_t* err, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaGetLastError();
}
}  // namespace attn
