// decode_noalloc.cu -- split-KV decode + merge for callers that cannot allocate
// device memory.
//
// attn_decode_split needs a caller-allocated buffer for the per-split partial
// results (part_o, part_lse) that attn_merge then combines.  Some callers
// cannot provide one: code running under a memory pool that has already
// reserved the device's memory, code that must not call cudaMalloc/cudaFree
// (both can synchronise the whole device), or plain C callers that have no
// device allocator at all.  attn_decode_noalloc keeps those partials in a
// fixed-size array of device memory that belongs to the library instead.
//
// The array below is part of this library's device code, so it is reserved on
// a GPU when that code is loaded there -- with CUDA's default lazy loading, at
// the library's first use on that device -- and stays reserved until the
// process exits.  All calls on a device share it: a call overwrites every entry
// it reads before reading it, so nothing has to start at zero, but two calls
// whose work overlaps on the GPU (e.g. on two streams) race on it.  The cached
// address below does not survive a cudaDeviceReset() of its device.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn.h"
#include "internal.h"

namespace {

// 24 MiB of fp32: part_o (B*Hq*n_splits*d floats) followed by part_lse
// (B*Hq*n_splits floats), each starting on a 256-byte boundary.
constexpr size_t kScratchBytes = size_t(24) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of this device's scratch array.  In host code the array's
// name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
int scratch_address(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

size_t round_up_256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" {

unsigned long long attn_decode_noalloc_scratch_bytes(void) { return kScratchBytes; }

int attn_decode_noalloc(const attn_bf16_t* q, const attn_bf16_t* kcache, const attn_bf16_t* vcache,
                        const int* kv_lens, int B, int Hq, int Hkv, int d, int max_kv, float scale,
                        int n_splits, int min_rows_per_split, void* o, float* lse, int o_dtype,
                        attn_stream_t stream) {
  // the argument rules of attn_decode_split (its partial buffers aside: they are
  // the scratch array) and of attn_merge, checked before the size and before any
  // CUDA call, so a malformed call is reported as such whatever its size
  int rc = attn::check_decode_split_args(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale,
                                         n_splits, min_rows_per_split, nullptr, nullptr, false);
  if (rc != ATTN_OK) return rc;
  rc = attn::check_merge_args(nullptr, nullptr, o, lse, B, Hq, n_splits, d, o_dtype, false);
  if (rc != ATTN_OK) return rc;
  if (B == 0) return ATTN_OK;
  const size_t rows = (size_t)B * (size_t)Hq * (size_t)n_splits;
  const size_t o_bytes = round_up_256(rows * (size_t)d * sizeof(float));
  const size_t lse_bytes = round_up_256(rows * sizeof(float));
  if (o_bytes + lse_bytes > kScratchBytes) return ATTN_ERR_SCRATCH_TOO_SMALL;
  float* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != ATTN_OK) return rc;
  float* part_o = scratch;
  float* part_lse = scratch + o_bytes / sizeof(float);
  rc = attn_decode_split(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale, n_splits,
                         min_rows_per_split, part_o, part_lse, stream);
  if (rc != ATTN_OK) return rc;
  return attn_merge(part_o, part_lse, o, lse, B, Hq, n_splits, d, o_dtype, stream);
}

}  // extern "C"
