"""Seeded synthetic inputs and the named workload shapes.

This module holds no attention arithmetic: it only draws i.i.d. N(0, 1)
values (fp32 from a seeded CPU generator, rounded to bf16 with
round-to-nearest-even) and KV lengths, with the shapes of the workloads the
engine is measured on.  Both the CUDA path and the fp64 oracle are fed from
here, so the two always see the same bf16 bits.

Workloads (names used throughout the tests and the benchmark):

* ``tiny_mha_causal``   B=1, Hq=Hkv=2, Sq=Skv=128, d=64, causal, scale 1/8, O fp32
* ``gqa_prefill_3314``  B=1, Hq=28, Hkv=4, Sq=Skv=3314, d=128, causal, scale 1/sqrt(128), O bf16
* ``gqa_decode_1641``   B=1, Hq=28, Hkv=4, one query token, KV length 1641, d=128,
                        8 splits (min 1 row per split), merged to O bf16 + LSE fp32
* ``mha_noncausal_4096_d{64,128,256,512}``  B=2, Hq=Hkv=16, S=4096, non-causal, scale 1/sqrt(d)
* ``ragged_gqa_decode_b64`` B=64, Hq=32, Hkv=8, d=128, KV lengths ~ U[512, 8192],
                        at most 4 splits of at least 1536 rows each (1 to 4 per
                        sequence, chosen by its length), O bf16 + LSE fp32
* ``gqa_prefill_3314_window1024_sink4`` the GQA prefill inputs, causal over a
                        1024-position sliding window plus 4 sink positions
* ``mqa_decode_b128_h128``  one-token decode, 128 query heads sharing one KV head
                        (B = 128, d = 128, lengths U[512, 8192])
* ``chunked_prefill_gqa_b8`` packed variable-length prefill against a KV cache:
                        B=8, Hq=28, Hkv=4, d=128, causal, 64-1024 new rows per
                        sequence after 0-3072 cached ones, O bf16 + LSE fp32
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class PrefillShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    d: int
    causal: bool
    scale: float
    out_dtype: str  # "f32" or "bf16"
    seed: int


@dataclass(frozen=True)
class DecodeShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    scale: float
    n_splits: int
    min_rows_per_split: int
    seed: int
    fixed_len: int | None = None          # every sequence this long, or
    len_range: tuple[int, int] | None = None  # lengths ~ U[lo, hi] from the seed
    out_dtype: str = "bf16"


TINY = PrefillShape("tiny_mha_causal", 1, 2, 2, 128, 128, 64, True, 1.0 / 8.0, "f32", 1001)
GQA_PREFILL = PrefillShape("gqa_prefill_3314", 1, 28, 4, 3314, 3314, 128, True,
                           1.0 / math.sqrt(128.0), "bf16", 1002)
GQA_DECODE = DecodeShape("gqa_decode_1641", 1, 28, 4, 128, 1.0 / math.sqrt(128.0), 8, 1, 1003,
                         fixed_len=1641)


def mha_sweep(d: int) -> PrefillShape:
    """The non-causal head-dim sweep (B=2, H=16, S=4096) at head dim d: 64, 128 and
    256 are the configured sweep, 512 extends it to the widest head the prefill takes."""
    return PrefillShape(f"mha_noncausal_4096_d{d}", 2, 16, 16, 4096, 4096, d, False,
                        1.0 / math.sqrt(float(d)), "bf16", 1000 + 4 * 10 + d // 64)


# split policy: 4 splits of at least 1536 rows (a sweep of 4/8/16 splits and
# 512-2048 minimum rows on one GB300: 223.9 us split + merge, 8 of 1024: 231.0)
RAGGED_DECODE = DecodeShape("ragged_gqa_decode_b64", 64, 32, 8, 128, 1.0 / math.sqrt(128.0), 4,
                            1536, 1005, len_range=(512, 8192))

# multi-query decode (one KV head for 128 query heads, the head count of the
# FMHA page's D2 workload), head dimension 128, ragged lengths as the GQA batch
MQA_DECODE = DecodeShape("mqa_decode_b128_h128", 128, 128, 1, 128, 1.0 / math.sqrt(128.0), 1,
                         1, 1008, len_range=(512, 8192))


# key splits of the multi-query decode on the tensor cores: (n_splits, min rows per
# split), 128-key multiples so a split is whole KV tiles
MQA_DECODE_SPLITS = (16, 512)


def decode_flops(kv_lens, Hq, d) -> int:
    """Algorithmic decode FLOPs: 4*d per (query head, cached key) pair."""
    total = int(torch.as_tensor(kv_lens).to(torch.int64).sum().item())
    return 4 * d * Hq * total


@dataclass(frozen=True)
class VarlenShape:
    """Packed chunked prefill: B sequences, each with Sq_b new query rows after a
    history of H_b cached tokens (L_b = H_b + Sq_b keys, the new rows last)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    causal: bool
    scale: float
    sq_range: tuple[int, int]    # new rows ~ U[lo, hi]
    hist_range: tuple[int, int]  # cached history ~ U[lo, hi]
    seed: int
    out_dtype: str = "bf16"


# a chunked-prefill batch of the 7B-class GQA shape: 8 sequences, 64-1024 new
# tokens each after 0-3072 cached ones
CHUNKED_PREFILL = VarlenShape("chunked_prefill_gqa_b8", 8, 28, 4, 128, True, 1.0 / math.sqrt(128.0),
                              (64, 1024), (0, 3072), 1006)


@dataclass(frozen=True)
class WindowShape:
    """Causal prefill over a sliding window of ``window`` positions plus ``n_sink``
    attention-sink positions, on the inputs of ``base``."""
    name: str
    base: PrefillShape
    window: int
    n_sink: int


# the GQA prefill shape with a 1024-position window and 4 sink positions
WINDOW_PREFILL = WindowShape("gqa_prefill_3314_window1024_sink4", GQA_PREFILL, 1024, 4)


def window_pairs(Sq: int, Skv: int, window: int, n_sink: int) -> int:
    """Admissible (query, key) pairs of one head of a windowed causal prefill."""
    total = 0
    for i in range(Sq):
        p = i + Skv - Sq
        if p < 0:
            continue
        hi = min(p, Skv - 1)
        lo = max(0, p - window + 1)
        win = max(0, hi - lo + 1)
        sinks = max(0, min(n_sink, hi + 1, lo))  # sink keys below the window
        total += win + sinks
    return total


def window_flops(s: WindowShape) -> int:
    """Algorithmic FLOPs: 4*d per admissible (query, key) pair."""
    b = s.base
    return 4 * b.d * b.B * b.Hq * window_pairs(b.Sq, b.Skv, s.window, s.n_sink)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    """i.i.d. N(0,1) drawn in fp32, then rounded to bf16 (RNE)."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def prefill_inputs(B, Hq, Hkv, Sq, Skv, d, seed):
    """Q [B,Sq,Hq,d], K/V [B,Skv,Hkv,d] bf16 on the CPU."""
    g = _gen(seed)
    q = randn_bf16((B, Sq, Hq, d), g)
    k = randn_bf16((B, Skv, Hkv, d), g)
    v = randn_bf16((B, Skv, Hkv, d), g)
    return q, k, v


def prefill_inputs_for(shape: PrefillShape):
    return prefill_inputs(shape.B, shape.Hq, shape.Hkv, shape.Sq, shape.Skv, shape.d, shape.seed)


def kv_lengths(B, lo, hi, seed) -> torch.Tensor:
    """Per-sequence KV lengths ~ U[lo, hi] (inclusive), int32."""
    g = _gen(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def decode_inputs(B, Hq, Hkv, d, kv_lens: torch.Tensor, seed, Lmax: int | None = None):
    """q [B,Hq,d], kcache/vcache [B,Lmax,Hkv,d] bf16 on the CPU."""
    if Lmax is None:
        Lmax = int(kv_lens.max().item()) if kv_lens.numel() else 0
    g = _gen(seed + 7919)
    q = randn_bf16((B, Hq, d), g)
    kc = randn_bf16((B, Lmax, Hkv, d), g)
    vc = randn_bf16((B, Lmax, Hkv, d), g)
    return q, kc, vc


def decode_inputs_for(shape: DecodeShape):
    if shape.fixed_len is not None:
        lens = torch.full((shape.B,), shape.fixed_len, dtype=torch.int32)
    else:
        lo, hi = shape.len_range
        lens = kv_lengths(shape.B, lo, hi, shape.seed)
    q, kc, vc = decode_inputs(shape.B, shape.Hq, shape.Hkv, shape.d, lens, shape.seed)
    return q, kc, vc, lens


def prefill_flops(B, Hq, Sq, Skv, d, causal) -> int:
    """Algorithmic FLOPs: 4*d per admissible (query, key) pair (2*d for QK^T, 2*d for PV)."""
    if causal:
        off = Skv - Sq
        pairs = 0
        # admissible keys of query i: j in [0, min(Skv, i + off + 1))
        for i in range(Sq):
            pairs += max(0, min(Skv, i + off + 1))
    else:
        pairs = Sq * Skv
    return 4 * d * B * Hq * pairs


def decode_kv_bytes(kv_lens, Hkv, d, elem_bytes=2) -> int:
    """Algorithmic K+V bytes: every cached row of every KV head read once."""
    total = int(torch.as_tensor(kv_lens).to(torch.int64).sum().item())
    return total * Hkv * d * elem_bytes * 2


def varlen_inputs(B, Hq, Hkv, d, sq: torch.Tensor, kv_lens: torch.Tensor, seed, max_kv: int | None = None):
    """Packed q [total_q,Hq,d], kcache/vcache [B,max_kv,Hkv,d] bf16 and cu_seqlens_q
    int32 [B+1] on the CPU, for new-row counts ``sq`` and key counts ``kv_lens``."""
    if max_kv is None:
        max_kv = int(kv_lens.max().item()) if kv_lens.numel() else 0
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(sq.to(torch.int64), 0).to(torch.int32)
    g = _gen(seed + 104729)
    q = randn_bf16((int(cu[-1].item()), Hq, d), g)
    kc = randn_bf16((B, max_kv, Hkv, d), g)
    vc = randn_bf16((B, max_kv, Hkv, d), g)
    return q, kc, vc, cu


def varlen_inputs_for(shape: VarlenShape):
    """(q, kcache, vcache, cu_seqlens_q, kv_lens) of a chunked-prefill workload."""
    sq = kv_lengths(shape.B, shape.sq_range[0], shape.sq_range[1], shape.seed)
    hist = kv_lengths(shape.B, shape.hist_range[0], shape.hist_range[1], shape.seed + 1)
    kv = (sq + hist).to(torch.int32)
    q, kc, vc, cu = varlen_inputs(shape.B, shape.Hq, shape.Hkv, shape.d, sq, kv, shape.seed)
    return q, kc, vc, cu, kv


def varlen_flops(cu: torch.Tensor, kv_lens: torch.Tensor, Hq: int, d: int, causal: bool) -> int:
    """Algorithmic FLOPs of a packed prefill: 4*d per admissible (query, key) pair."""
    total = 0
    for b in range(kv_lens.numel()):
        sq = int(cu[b + 1] - cu[b])
        L = int(kv_lens[b])
        if causal:
            off = L - sq
            pairs = sum(max(0, min(L, i + off + 1)) for i in range(sq))
        else:
            pairs = sq * L
        total += pairs
    return 4 * d * Hq * total
