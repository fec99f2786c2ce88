// decode.cu -- one-token GQA decode on CUDA cores: split-KV partials and the
// LSE-weighted merge.
//
// What one split computes follows "66 . D2: explicit K+V register staging",
// section 3.2: for the rows [lo, hi) of one sequence and one KV head, every
// query head of the GQA group takes the score s = (q . k) * scale, keeps a
// running max, a running sum and a running O, and rescales both by
// exp(m_old - m_new) when the max grows.  Section 2.2 of that page moves the
// K and V loads ahead of the exp/shuffle dependency chain; here the same idea
// is carried by the GB300 copy engine: one producer warp issues TMA tile loads
// (32 rows of K and of V per stage) into a shared-memory ring, so the loads of
// later tiles are in flight while the consumer warps work on earlier ones.
//
// Work mapping (per CTA = one (batch, KV head, split)):
//   * warp 4 (producer): TMA loads of K and V tiles into the ring;
//   * warps 0..3 (consumers): warp w owns tiles w, w+4, w+8, ... of the split.
//     Scores: lane = row of the tile, the whole head dim of that row from
//     shared memory against every query head of the group (q kept in shared
//     memory in fp32, pre-multiplied by scale * log2(e)).  Softmax: warp
//     max by shuffles, exp2 on the MUFU.  P.V: lane = d/32 consecutive dims,
//     one V row per step, p broadcast from shared memory.
//   * at the end the four warps' partial (m, l, O) are merged through shared
//     memory and the split's normalised O and its LSE are written.
// Everything is fp32 on CUDA cores; no tensor cores.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kNumConsumerWarps = 4;
constexpr int kDecodeThreads = (kNumConsumerWarps + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, int GMAX>
struct DecodeCfg {
  static constexpr int kTile = kDecodeTileRows;        // rows per stage
  static constexpr int kPanels = D / 64;               // 128-byte swizzled panels per row
  static constexpr int kPanelBytes = kTile * 128;      // one panel of one tile
  static constexpr int kKBytes = kPanels * kPanelBytes;
  static constexpr int kStageBytes = 2 * kKBytes;      // K then V
  static constexpr int kStages = kNumConsumerWarps;    // one stage per consumer warp
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kQBytes = GMAX * D * 4;                             // fp32 q
  static constexpr int kPBytes = kNumConsumerWarps * kTile * GMAX * 4;     // p per warp [row][g]
  static constexpr int kCombBytes = kNumConsumerWarps * GMAX * (D + 2) * 4;
  static_assert(kCombBytes <= kRingBytes, "combine area must fit in the ring");
  static constexpr int kBarOffset = kRingBytes + kQBytes + kPBytes;
  static constexpr int kSmemBytes = kBarOffset + 2 * kStages * 8 + 16 + 1024;  // + align slack
};

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

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

__device__ __forceinline__ void consumer_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kNumConsumerWarps * 32) : "memory");
}

template <int D, int GMAX>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const uint16_t* __restrict__ q,
                        const int* __restrict__ kv_lens, float* __restrict__ part_o,
                        float* __restrict__ part_lse, int Hq, int Hkv, int max_kv, int n_splits,
                        int min_rows, float scale, uint32_t* err) {
  using C = DecodeCfg<D, GMAX>;
  constexpr int DPL = D / 32;  // output dims per lane in the P.V phase
  const int s_idx = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- split bounds: chunk = max(ceil(L / n_splits), min_rows) ----
  int L = kv_lens[b];
  L = L < 0 ? 0 : (L > max_kv ? max_kv : L);
  long long chunk = ((long long)L + n_splits - 1) / n_splits;
  if (chunk < min_rows) chunk = min_rows;
  if (chunk < 1) chunk = 1;
  long long lo_ll = (long long)s_idx * chunk, hi_ll = lo_ll + chunk;
  const int lo = (int)(lo_ll < L ? lo_ll : L), hi = (int)(hi_ll < L ? hi_ll : L);

  if (lo >= hi) {  // empty split: o = 0, lse = -inf; nothing is read
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
      const int g = i / D, t = i % D;
      const size_t row = ((size_t)b * Hq + (size_t)hk * G + g) * n_splits + s_idx;
      part_o[row * D + t] = 0.f;
      if (t == 0) part_lse[row] = -INFINITY;
    }
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* qs = reinterpret_cast<float*>(smem + C::kRingBytes);                   // [GMAX][D]
  float* pbuf = reinterpret_cast<float*>(smem + C::kRingBytes + C::kQBytes);    // [warp][row][GMAX]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* empty = full + C::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::kStages);

  const int T = (hi - lo + C::kTile - 1) / C::kTile;  // tiles in this split

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // q of the group, fp32, pre-scaled into the log2 domain
  const float qscale = scale * kLog2e;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int g = i / D, t = i % D;
    const uint16_t raw = q[((size_t)b * Hq + (size_t)hk * G + g) * D + t];
    qs[g * D + t] = __uint_as_float((uint32_t)raw << 16) * qscale;
  }
  for (int i = threadIdx.x; i < (GMAX - G) * D; i += blockDim.x) qs[G * D + i] = 0.f;
  __syncthreads();

  if (warp == kNumConsumerWarps) {
    // ================= producer warp =================
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol = l2_policy_evict_first();
      int t = 0;
      for (; t < T; ++t) {
        const int s = t % C::kStages, k = t / C::kStages;
        if (!mbar_wait(&empty[s], (k & 1) ^ 1, err, abort_flag)) break;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        uint8_t* kdst = ring + s * C::kStageBytes;
        uint8_t* vdst = kdst + C::kKBytes;
        const int row = lo + t * C::kTile;
#pragma unroll
        for (int p = 0; p < C::kPanels; ++p) {
          tma_load_4d_hint(kdst + p * C::kPanelBytes, &tm_k, &full[s], p * 64, hk, row, b, pol);
          tma_load_4d_hint(vdst + p * C::kPanelBytes, &tm_v, &full[s], p * 64, hk, row, b, pol);
        }
      }
      if (t < T) {
        // aborted: let the copies already issued land before the CTA exits
        for (int u = (t - C::kStages > 0 ? t - C::kStages : 0); u < t; ++u)
          mbar_wait(&full[u % C::kStages], (u / C::kStages) & 1, nullptr, nullptr, 100000000ull);
      }
    }
    return;  // the producer takes no part in the combine
  }

  // ================= consumer warps =================
  float m[GMAX], lsum[GMAX], o[GMAX][DPL];
#pragma unroll
  for (int g = 0; g < GMAX; ++g) {
    m[g] = -INFINITY;
    lsum[g] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
  }
  float* pw = pbuf + warp * C::kTile * GMAX;

  bool ok = true;
  for (int t = warp; t < T; t += kNumConsumerWarps) {
    const int s = t % C::kStages, k = t / C::kStages;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], k & 1, err, abort_flag))) {
      ok = false;
      break;
    }
    const uint8_t* kt = ring + s * C::kStageBytes;
    const uint8_t* vt = kt + C::kKBytes;
    const int row0 = lo + t * C::kTile;
    const int nrows = min(C::kTile, hi - row0);

    // ---- scores: lane = row ----
    float acc[GMAX];
#pragma unroll
    for (int g = 0; g < GMAX; ++g) acc[g] = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const int p = c >> 3, cc = c & 7;
      const uint4 kv = *reinterpret_cast<const uint4*>(kt + p * C::kPanelBytes + lane * 128 +
                                                       ((cc ^ (lane & 7)) << 4));
      const float k0 = bf16lo(kv.x), k1 = bf16hi(kv.x), k2 = bf16lo(kv.y), k3 = bf16hi(kv.y);
      const float k4 = bf16lo(kv.z), k5 = bf16hi(kv.z), k6 = bf16lo(kv.w), k7 = bf16hi(kv.w);
#pragma unroll
      for (int g = 0; g < GMAX; ++g) {
        if (g < G) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + g * D + c * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qs + g * D + c * 8 + 4);
          float a = acc[g];
          a = fmaf(qa.x, k0, a);
          a = fmaf(qa.y, k1, a);
          a = fmaf(qa.z, k2, a);
          a = fmaf(qa.w, k3, a);
          a = fmaf(qb.x, k4, a);
          a = fmaf(qb.y, k5, a);
          a = fmaf(qb.z, k6, a);
          a = fmaf(qb.w, k7, a);
          acc[g] = a;
        }
      }
    }
    const bool valid = lane < nrows;

    // ---- online softmax per query head (log2 domain) ----
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
      if (g < G) {
        const float sv = valid ? acc[g] : -INFINITY;
        const float tmax = warp_max(sv);  // finite: every tile has >= 1 valid row
        const float m_new = fmaxf(m[g], tmax);
        const float corr = ex2_approx(m[g] - m_new);  // m = -inf -> 0
        const float pv = ex2_approx(sv - m_new);      // invalid -> 0
        lsum[g] = fmaf(lsum[g], corr, pv);           // per-lane partial sum
        m[g] = m_new;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[g][e] *= corr;
        pw[lane * GMAX + g] = pv;
      }
    }
    __syncwarp();

    // ---- O += P V: lane = DPL consecutive dims ----
#pragma unroll 2
    for (int r = 0; r < nrows; ++r) {
      float vf[DPL];
      if constexpr (D == 64) {
        const uint32_t x = *reinterpret_cast<const uint32_t*>(
            vt + r * 128 + (((lane >> 2) ^ (r & 7)) << 4) + (lane & 3) * 4);
        vf[0] = bf16lo(x);
        vf[1] = bf16hi(x);
      } else if constexpr (D == 128) {
        const uint2 x = *reinterpret_cast<const uint2*>(
            vt + (lane >> 4) * C::kPanelBytes + r * 128 + ((((lane & 15) >> 1) ^ (r & 7)) << 4) +
            (lane & 1) * 8);
        vf[0] = bf16lo(x.x);
        vf[1] = bf16hi(x.x);
        vf[2] = bf16lo(x.y);
        vf[3] = bf16hi(x.y);
      } else {
        const uint4 x = *reinterpret_cast<const uint4*>(vt + (lane >> 3) * C::kPanelBytes + r * 128 +
                                                        (((lane & 7) ^ (r & 7)) << 4));
        vf[0] = bf16lo(x.x);
        vf[1] = bf16hi(x.x);
        vf[2] = bf16lo(x.y);
        vf[3] = bf16hi(x.y);
        vf[4] = bf16lo(x.z);
        vf[5] = bf16hi(x.z);
        vf[6] = bf16lo(x.w);
        vf[7] = bf16hi(x.w);
      }
      const float* pr = pw + r * GMAX;
#pragma unroll
      for (int g4 = 0; g4 < GMAX; g4 += 4) {
        if (g4 < G) {
          const float4 p4 = *reinterpret_cast<const float4*>(pr + g4);
          const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[g4 + gg][e] = fmaf(pp[gg], vf[e], o[g4 + gg][e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- combine the consumer warps' partials through shared memory ----
  consumer_bar_sync();  // every consumer is done with the ring
  float* comb = reinterpret_cast<float*>(ring);  // [warp][g][D + 2]: o[0..D), m, l
#pragma unroll
  for (int g = 0; g < GMAX; ++g) {
    if (g < G) {
      const float lw = warp_sum(lsum[g]);
      float* cw = comb + (warp * GMAX + g) * (D + 2);
#pragma unroll
      for (int e = 0; e < DPL; ++e) cw[lane * DPL + e] = o[g][e];
      if (lane == 0) {
        cw[D] = m[g];
        cw[D + 1] = lw;
      }
    }
  }
  consumer_bar_sync();
  if (!ok || *abort_flag) return;
  for (int i = threadIdx.x; i < G * D; i += kNumConsumerWarps * 32) {
    const int g = i / D, t = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kNumConsumerWarps; ++w) M = fmaxf(M, comb[(w * GMAX + g) * (D + 2) + D]);
    float Lsum = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kNumConsumerWarps; ++w) {
      const float* cw = comb + (w * GMAX + g) * (D + 2);
      const float f = ex2_approx(cw[D] - M);  // warps without tiles: m = -inf -> 0
      Lsum = fmaf(cw[D + 1], f, Lsum);
      acc = fmaf(cw[t], f, acc);
    }
    const size_t row = ((size_t)b * Hq + (size_t)hk * G + g) * n_splits + s_idx;
    part_o[row * D + t] = acc / Lsum;
    if (t == 0) part_lse[row] = (M + log2f(Lsum)) * kLn2;
  }
}

template <int D>
__global__ void __launch_bounds__(128)
    merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, void* o,
                 float* __restrict__ lse, int rows, int n_splits, int o_bf16) {
  constexpr int DPL = D / 32;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* pl = part_lse + (size_t)row * n_splits;
  const float* po = part_o + (size_t)row * n_splits * D;
  float M = -INFINITY;
  for (int s = lane; s < n_splits; s += 32) M = fmaxf(M, pl[s]);
  M = warp_max(M);
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const float ls = pl[s];
      if (ls == -INFINITY) continue;  // empty split: its part_o is not read
      const float w = ex2_approx((ls - M) * kLog2e);
      wsum += w;
      const float* src = po + (size_t)s * D + lane * DPL;
#pragma unroll
      for (int e = 0; e < DPL; e += 2) {
        const float2 x = *reinterpret_cast<const float2*>(src + e);
        acc[e] = fmaf(w, x.x, acc[e]);
        acc[e + 1] = fmaf(w, x.y, acc[e + 1]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  if (o_bf16) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(o) + (size_t)row * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; e += 2) {
      *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    }
  } else {
    float* dst = reinterpret_cast<float*>(o) + (size_t)row * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; e += 2) {
      *reinterpret_cast<float2*>(dst + e) = make_float2(acc[e] * inv, acc[e + 1] * inv);
    }
  }
  if (lane == 0) lse[row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

template <int D, int GMAX>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
  using C = DecodeCfg<D, GMAX>;
  auto kern = decode_split_kernel<D, GMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_splits, a.Hkv, a.B);
  kern<<<grid, kDecodeThreads, C::kSmemBytes, stream>>>(a.tm_k, a.tm_v, a.q, a.kv_lens, a.part_o,
                                                         a.part_lse, a.Hq, a.Hkv, a.max_kv,
                                                         a.n_splits, a.min_rows, a.scale, a.err);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_g(const DecodeArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  if (G <= 4) return launch_decode_t<D, 4>(a, stream);
  if (G <= 8) return launch_decode_t<D, 8>(a, stream);
  return launch_decode_t<D, 16>(a, stream);
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
