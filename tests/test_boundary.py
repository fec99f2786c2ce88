"""The C-ABI library: it loads, exports every declared symbol, and rejects bad
arguments on the host (no GPU needed: validation runs before any CUDA call)."""
import ctypes
import os
import re

import pytest

import attention_forward_tcgen05_gb300 as attn
from attention_forward_tcgen05_gb300 import build as attn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    attn_build.build()
    return attn.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*|unsigned long long)\s+(attn_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert len(syms) >= 7
    for s in syms:
        assert hasattr(lib, s), f"{s} declared in attn.h but not exported"


def test_version_and_strerror(lib):
    assert attn.attn_version() >= 10000
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert attn.attn_strerror(code)
    assert attn.attn_strerror(12345) == "unknown status"


N = None  # null pointer
P = ctypes.c_void_p(16)  # an aligned non-null dummy (never dereferenced: validation fails first)
M = ctypes.c_void_p(18)  # misaligned


def test_prefill_validation(lib):
    f = attn.attn_prefill_fwd
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 96, 1, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED  # d
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 64, 1, 0.5, 7, N) == attn.ATTN_ERR_UNSUPPORTED  # dtype
    assert f(P, P, P, P, P, 1, 3, 2, 4, 4, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # Hq % Hkv
    assert f(P, P, P, P, P, -1, 2, 2, 4, 4, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 64, 1, 0.0, 0, N) == attn.ATTN_ERR_INVALID_ARG  # scale
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 64, 1, float("nan"), 0, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(N, P, P, P, P, 1, 2, 2, 4, 4, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # null q
    assert f(P, P, M, P, P, 1, 2, 2, 4, 4, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # misaligned v
    assert f(N, N, N, N, N, 0, 2, 2, 4, 4, 64, 1, 0.5, 0, N) == attn.ATTN_OK  # empty batch: no-op
    assert f(N, N, N, N, N, 2, 2, 2, 0, 4, 64, 1, 0.5, 0, N) == attn.ATTN_OK  # no queries: no-op
    assert f(N, N, N, N, N, 0, 2, 2, 4, 4, 512, 1, 0.5, 0, N) == attn.ATTN_OK  # d = 512 accepted
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 1024, 1, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED


def test_head_dim_512_only_on_the_plain_prefill(lib):
    """d = 512 runs through attn_prefill_fwd; the other entry points refuse it."""
    assert attn.attn_prefill_window(P, P, P, P, P, 1, 2, 2, 4, 4, 512, 8, 0, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_prefill_packed(P, P, P, P, P, 1, 8, 1, 4, 4, 512, 1, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_prefill_varlen(P, P, P, P, P, P, P, 2, 2, 2, 10, 8, 16, 512, 1, 0.5, 0, N) == \
        attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_decode_split(P, P, P, P, 1, 8, 2, 512, 10, 0.1, 4, 1, P, P, N) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_decode_packed(P, P, P, P, 2, 8, 1, 512, 16, 0.5, P, P, 0, N) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_merge(P, P, P, P, 1, 4, 8, 512, 1, N) == attn.ATTN_ERR_UNSUPPORTED


def test_prefill_window_validation(lib):
    f = attn.attn_prefill_window
    #      q  k  v  o  lse B  Hq Hkv Sq Skv d  win sink scale dtype stream
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 96, 8, 0, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED  # d
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 64, 8, 0, 0.5, 5, N) == attn.ATTN_ERR_UNSUPPORTED  # dtype
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 64, 0, 0, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # window 0
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 64, -3, 0, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # window < 0
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 64, 8, -1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # n_sink < 0
    assert f(P, P, P, P, P, 1, 3, 2, 4, 4, 64, 8, 0, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # Hq % Hkv
    assert f(P, P, P, P, P, 1, 2, 2, 4, 4, 64, 8, 0, -1.0, 0, N) == attn.ATTN_ERR_INVALID_ARG  # scale
    assert f(P, M, P, P, P, 1, 2, 2, 4, 4, 64, 8, 0, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # misaligned k
    assert f(N, N, N, N, N, 0, 2, 2, 4, 4, 64, 8, 4, 0.5, 0, N) == attn.ATTN_OK  # empty batch
    assert f(N, N, N, N, N, 2, 2, 2, 0, 4, 64, 8, 4, 0.5, 0, N) == attn.ATTN_OK  # no queries


def test_prefill_varlen_validation(lib):
    f = attn.attn_prefill_varlen
    #      q  kc vc o  lse cu kv  B  Hq Hkv tot msq mkv d  causal scale dtype stream
    assert f(P, P, P, P, P, P, P, 2, 2, 2, 10, 8, 16, 96, 1, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED  # d
    assert f(P, P, P, P, P, P, P, 2, 2, 2, 10, 8, 16, 64, 1, 0.5, 9, N) == attn.ATTN_ERR_UNSUPPORTED  # dtype
    assert f(P, P, P, P, P, P, P, 2, 3, 2, 10, 8, 16, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # Hq % Hkv
    assert f(P, P, P, P, P, P, P, 2, 2, 2, -1, 8, 16, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # total_q
    assert f(P, P, P, P, P, P, P, 2, 2, 2, 10, 8, -1, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # max_kv
    assert f(P, P, P, P, P, P, P, 2, 2, 2, 10, 8, 16, 64, 1, -0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # scale
    assert f(P, P, P, P, P, N, P, 2, 2, 2, 10, 8, 16, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # null cu
    assert f(P, P, P, P, P, P, ctypes.c_void_p(18), 2, 2, 2, 10, 8, 16, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # kv_lens misaligned
    assert f(P, M, P, P, P, P, P, 2, 2, 2, 10, 8, 16, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # kcache misaligned
    assert f(N, N, N, N, N, N, N, 0, 2, 2, 10, 8, 16, 64, 1, 0.5, 0, N) == attn.ATTN_OK  # empty batch
    assert f(N, N, N, N, N, N, N, 3, 2, 2, 0, 0, 16, 64, 1, 0.5, 0, N) == attn.ATTN_OK  # no query rows


def test_prefill_varlen_window_validation(lib):
    f = attn.attn_prefill_varlen_window
    #      q  kc vc o  lse cu kv  B  Hq Hkv tot msq mkv d  win sink scale dtype stream
    assert f(P, P, P, P, P, P, P, 2, 2, 2, 10, 8, 16, 96, 4, 0, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED  # d
    assert f(P, P, P, P, P, P, P, 2, 2, 2, 10, 8, 16, 64, 0, 0, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # window
    assert f(P, P, P, P, P, P, P, 2, 2, 2, 10, 8, 16, 64, 4, -2, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # n_sink
    assert f(P, P, P, P, P, N, P, 2, 2, 2, 10, 8, 16, 64, 4, 0, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # null cu
    assert f(P, P, P, P, P, P, P, 2, 3, 2, 10, 8, 16, 64, 4, 0, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # Hq % Hkv
    assert f(N, N, N, N, N, N, N, 0, 2, 2, 10, 8, 16, 64, 4, 0, 0.5, 0, N) == attn.ATTN_OK  # empty batch


def test_packed_validation(lib):
    f = attn.attn_prefill_packed
    #      q  k  v  o  lse B  Hq Hkv Sq Skv d    causal scale dtype stream
    assert f(P, P, P, P, P, 1, 8, 1, 4, 4, 256, 1, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED  # d = 256
    assert f(P, P, P, P, P, 1, 6, 2, 4, 4, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED  # G = 3
    assert f(P, P, P, P, P, 1, 256, 1, 4, 4, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_UNSUPPORTED  # G = 256
    assert f(P, P, P, P, P, 1, 6, 4, 4, 4, 64, 1, 0.5, 0, N) == attn.ATTN_ERR_INVALID_ARG  # Hq % Hkv
    assert f(N, N, N, N, N, 0, 8, 1, 4, 4, 64, 1, 0.5, 0, N) == attn.ATTN_OK  # empty batch
    g = attn.attn_decode_packed
    #      q  kc vc kv  B  Hq Hkv d   mkv scale o  lse dtype stream
    assert g(P, P, P, P, 2, 8, 1, 96, 16, 0.5, P, P, 0, N) == attn.ATTN_ERR_UNSUPPORTED  # d
    assert g(P, P, P, P, 2, 8, 1, 64, 16, 0.5, P, P, 3, N) == attn.ATTN_ERR_UNSUPPORTED  # dtype
    assert g(P, P, P, P, 2, 256, 1, 64, 16, 0.5, P, P, 0, N) == attn.ATTN_ERR_UNSUPPORTED  # G = 256
    assert g(P, P, P, N, 2, 8, 1, 64, 16, 0.5, P, P, 0, N) == attn.ATTN_ERR_INVALID_ARG  # null kv_lens
    assert g(P, P, P, M, 2, 8, 1, 64, 16, 0.5, P, P, 0, N) == attn.ATTN_ERR_INVALID_ARG  # misaligned kv_lens
    assert g(P, P, P, P, 2, 8, 1, 64, -1, 0.5, P, P, 0, N) == attn.ATTN_ERR_INVALID_ARG  # max_kv
    assert g(P, P, P, P, 2, 8, 1, 64, 16, 0.0, P, P, 0, N) == attn.ATTN_ERR_INVALID_ARG  # scale
    assert g(N, N, N, N, 0, 8, 1, 64, 16, 0.5, N, N, 0, N) == attn.ATTN_OK  # empty batch


def test_split_packed_validation(lib):
    f = attn.attn_decode_split_packed
    #      q  kc vc kv  B  Hq Hkv d   mkv scale ns mr po pl stream
    assert f(P, P, P, P, 2, 8, 1, 256, 16, 0.5, 4, 1, P, P, N) == attn.ATTN_ERR_UNSUPPORTED  # d
    assert f(P, P, P, P, 2, 256, 1, 64, 16, 0.5, 4, 1, P, P, N) == attn.ATTN_ERR_UNSUPPORTED  # G = 256
    assert f(P, P, P, P, 2, 8, 1, 64, 16, 0.5, 0, 1, P, P, N) == attn.ATTN_ERR_INVALID_ARG  # n_splits
    assert f(P, P, P, P, 2, 8, 1, 64, 16, 0.5, 4, -1, P, P, N) == attn.ATTN_ERR_INVALID_ARG  # min rows
    assert f(P, P, P, P, 2, 8, 1, 64, 16, 0.5, 4, 1, N, P, N) == attn.ATTN_ERR_INVALID_ARG  # null part_o
    assert f(P, P, P, P, 2, 8, 1, 64, 16, 0.5, 4, 1, P, M, N) == attn.ATTN_ERR_INVALID_ARG  # part_lse align
    assert f(N, N, N, N, 0, 8, 1, 64, 16, 0.5, 4, 1, N, N, N) == attn.ATTN_OK  # empty batch


def test_decode_and_merge_validation(lib):
    f = attn.attn_decode_split
    assert f(P, P, P, P, 1, 28, 4, 96, 10, 0.1, 8, 1, P, P, N) == attn.ATTN_ERR_UNSUPPORTED
    assert f(P, P, P, P, 1, 28, 5, 128, 10, 0.1, 8, 1, P, P, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, 1, 258, 2, 128, 10, 0.1, 8, 1, P, P, N) == attn.ATTN_ERR_INVALID_ARG  # G > 128
    assert f(P, P, P, P, 1, 28, 4, 128, 10, 0.1, 0, 1, P, P, N) == attn.ATTN_ERR_INVALID_ARG  # n_splits
    assert f(P, P, P, P, 1, 28, 4, 128, 0, 0.1, 8, 1, P, P, N) == attn.ATTN_ERR_INVALID_ARG  # max_kv
    assert f(P, P, P, N, 1, 28, 4, 128, 10, 0.1, 8, 1, P, P, N) == attn.ATTN_ERR_INVALID_ARG  # lens
    # one CTA per (sequence, KV head, split): more than 2^31 - 1 is refused up front
    assert f(P, P, P, P, 1 << 20, 4, 4, 64, 1, 0.1, 1024, 1, P, P, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(N, N, N, N, 0, 28, 4, 128, 10, 0.1, 8, 1, N, N, N) == attn.ATTN_OK
    g = attn.attn_merge
    assert g(P, P, P, P, 1, 4, 8, 100, 1, N) == attn.ATTN_ERR_UNSUPPORTED
    assert g(P, P, P, P, 1, 4, 0, 128, 1, N) == attn.ATTN_ERR_INVALID_ARG
    assert g(P, P, M, P, 1, 4, 8, 128, 1, N) == attn.ATTN_ERR_INVALID_ARG
    assert g(N, N, N, N, 0, 4, 8, 128, 1, N) == attn.ATTN_OK


def test_fused_decode_validation(lib):
    """attn_decode takes the rules of attn_decode_split and attn_merge, and needs a
    4-byte aligned counter buffer."""
    f = attn.attn_decode
    C = ctypes.c_void_p(20)  # 4-byte aligned counters
    #      q  kc vc kv B  Hq Hkv d    mkv scale ns mr po pl o  lse dtype ctr stream
    assert f(P, P, P, P, 1, 28, 4, 128, 10, 0.1, 8, 1, P, P, P, P, 1, N, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, 1, 28, 4, 128, 10, 0.1, 8, 1, P, P, P, P, 1, M, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, 1, 28, 4, 96, 10, 0.1, 8, 1, P, P, P, P, 1, C, N) == attn.ATTN_ERR_UNSUPPORTED
    assert f(P, P, P, P, 1, 28, 4, 128, 10, 0.1, 8, 1, P, P, P, P, 7, C, N) == attn.ATTN_ERR_UNSUPPORTED
    assert f(P, P, P, P, 1, 258, 2, 128, 10, 0.1, 8, 1, P, P, P, P, 1, C, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, 1, 28, 4, 128, 10, 0.1, 0, 1, P, P, P, P, 1, C, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, 1, 28, 4, 128, 10, 0.1, 8, 1, N, P, P, P, 1, C, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, 1, 28, 4, 128, 10, 0.1, 8, 1, P, P, M, P, 1, C, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, 1, 28, 4, 128, 10, 0.1, 8, 1, P, P, P, N, 1, C, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(N, N, N, N, 0, 28, 4, 128, 10, 0.1, 8, 1, N, N, N, N, 1, N, N) == attn.ATTN_OK


def test_debug_wait_limits(lib):
    assert attn.attn_debug_wait_timeout(10, N) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_debug_wait_timeout(10**11, N) == attn.ATTN_ERR_INVALID_ARG


def test_noalloc_validation(lib):
    """attn_decode_noalloc checks its arguments by the rules of attn_decode_split and
    attn_merge first, and the size of its problem against the static scratch after
    them: a malformed call is reported as malformed whatever its size."""
    f = attn.attn_decode_noalloc
    limit = attn.attn_decode_noalloc_scratch_bytes()
    assert limit == 24 << 20
    B, Hq, Hkv, d, n_splits = 64, 32, 8, 128, 32  # partials of 33.8 MB: beyond the scratch
    assert B * Hq * n_splits * (d + 1) * 4 > limit
    #      q  kc vc kv  B  Hq  Hkv  d  mkv scale  ns  mr o  lse dtype stream
    assert f(P, P, P, P, B, Hq, Hkv, d, 16, 0.1, n_splits, 1, P, P, attn.ATTN_BF16, N) == \
        attn.ATTN_ERR_SCRATCH_TOO_SMALL
    # oversized and malformed: the malformation is what is reported
    assert f(P, P, P, P, B, Hq, Hkv, d, 16, float("nan"), n_splits, 1, P, P, 1, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, M, P, P, B, Hq, Hkv, d, 16, 0.1, n_splits, 1, P, P, 1, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, B, Hq, Hkv, d, 16, 0.1, n_splits, 1, M, P, 1, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, B, Hq, Hkv, d, 16, 0.1, n_splits, 1, P, N, 1, N) == attn.ATTN_ERR_INVALID_ARG
    assert f(P, P, P, P, B, Hq, Hkv, 96, 16, 0.1, n_splits, 1, P, P, 1, N) == attn.ATTN_ERR_UNSUPPORTED
    assert f(P, P, P, P, B, Hq, Hkv, d, 16, 0.1, n_splits, 1, P, P, 5, N) == attn.ATTN_ERR_UNSUPPORTED
    assert f(P, P, P, P, B, 258, 2, d, 16, 0.1, n_splits, 1, P, P, 1, N) == attn.ATTN_ERR_INVALID_ARG  # G > 128
    assert f(P, P, P, P, B, Hq, Hkv, d, 16, 0.1, 2000, 1, P, P, 1, N) == attn.ATTN_ERR_INVALID_ARG  # n_splits
    # the rules shared with attn_decode_split on a problem that fits
    assert f(P, P, P, N, 2, 8, 2, 64, 16, 0.1, 4, 1, P, P, 1, N) == attn.ATTN_ERR_INVALID_ARG  # null kv_lens
    assert f(N, N, N, N, 0, 8, 2, 64, 16, 0.1, 4, 1, N, N, 1, N) == attn.ATTN_OK  # empty batch
