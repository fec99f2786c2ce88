"""ctypes binding of libattn.so (the C ABI in include/attn.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  The raw entry points keep the C names and argument
order; the torch helpers below allocate outputs with torch and pass device
pointers and the current CUDA stream.  If the library is missing this module
raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_CUDA = -3
ATTN_ERR_DEVICE_TIMEOUT = -4
ATTN_ERR_SCRATCH_TOO_SMALL = -5
ATTN_ERR_DEVICE_INPUT = -6
ATTN_F32 = 0
ATTN_BF16 = 1

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({attn_strerror(status)})")


def load(path: str | None = None):
    """Load libattn.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        vp, i, f, ull = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong
        lib.attn_prefill_fwd.argtypes = [vp, vp, vp, vp, vp] + [i] * 7 + [f, i, vp]
        lib.attn_prefill_varlen.argtypes = [vp] * 7 + [i] * 8 + [f, i, vp]
        lib.attn_prefill_window.argtypes = [vp] * 5 + [i] * 8 + [f, i, vp]
        lib.attn_prefill_varlen_window.argtypes = [vp] * 7 + [i] * 9 + [f, i, vp]
        lib.attn_prefill_packed.argtypes = [vp] * 5 + [i] * 7 + [f, i, vp]
        lib.attn_decode_packed.argtypes = [vp] * 4 + [i] * 5 + [f, vp, vp, i, vp]
        lib.attn_decode_split_packed.argtypes = [vp] * 4 + [i] * 5 + [f, i, i, vp, vp, vp]
        lib.attn_decode_split.argtypes = [vp, vp, vp, vp] + [i] * 5 + [f, i, i, vp, vp, vp]
        lib.attn_merge.argtypes = [vp, vp, vp, vp] + [i] * 5 + [vp]
        lib.attn_decode.argtypes = [vp] * 4 + [i] * 5 + [f, i, i, vp, vp, vp, vp, i, vp, vp]
        lib.attn_sync_check.argtypes = [vp]
        lib.attn_strerror.argtypes = [i]
        lib.attn_strerror.restype = ctypes.c_char_p
        lib.attn_version.argtypes = []
        lib.attn_debug_wait_timeout.argtypes = [ull, vp]
        lib.attn_prefill_schedule.argtypes = [i] * 5 + [vp, vp, i]
        lib.attn_decode_noalloc.argtypes = [vp, vp, vp, vp] + [i] * 5 + [f, i, i, vp, vp, i, vp]
        lib.attn_decode_noalloc_scratch_bytes.argtypes = []
        lib.attn_decode_noalloc_scratch_bytes.restype = ull
        for name in ("attn_prefill_fwd", "attn_prefill_varlen", "attn_prefill_window",
                     "attn_prefill_varlen_window", "attn_prefill_packed", "attn_decode_packed",
                     "attn_decode_split_packed",
                     "attn_decode_split", "attn_merge", "attn_decode",
                     "attn_sync_check",
                     "attn_version", "attn_debug_wait_timeout", "attn_decode_noalloc",
                     "attn_prefill_schedule"):
            getattr(lib, name).restype = i
        _lib = lib
        return lib


# ------------------------------------------------------------------ raw C ABI
def attn_prefill_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, causal, scale, o_dtype, stream) -> int:
    return load().attn_prefill_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, int(causal),
                                   float(scale), o_dtype, stream)


def attn_prefill_packed(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, causal, scale, o_dtype, stream) -> int:
    return load().attn_prefill_packed(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, int(causal),
                                      float(scale), o_dtype, stream)


def attn_decode_packed(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale, o, lse, o_dtype,
                       stream) -> int:
    return load().attn_decode_packed(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, float(scale),
                                     o, lse, o_dtype, stream)


def attn_decode_split_packed(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale, n_splits,
                             min_rows_per_split, part_o, part_lse, stream) -> int:
    return load().attn_decode_split_packed(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv,
                                           float(scale), n_splits, min_rows_per_split, part_o, part_lse,
                                           stream)


def attn_prefill_window(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, window, n_sink, scale, o_dtype,
                        stream) -> int:
    return load().attn_prefill_window(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, int(window),
                                      int(n_sink), float(scale), o_dtype, stream)


def attn_prefill_varlen(q, kcache, vcache, o, lse, cu_seqlens_q, kv_lens, B, Hq, Hkv, total_q,
                        max_sq, max_kv, d, causal, scale, o_dtype, stream) -> int:
    return load().attn_prefill_varlen(q, kcache, vcache, o, lse, cu_seqlens_q, kv_lens, B, Hq, Hkv,
                                      total_q, max_sq, max_kv, d, int(causal), float(scale), o_dtype,
                                      stream)


def attn_prefill_varlen_window(q, kcache, vcache, o, lse, cu_seqlens_q, kv_lens, B, Hq, Hkv,
                               total_q, max_sq, max_kv, d, window, n_sink, scale, o_dtype,
                               stream) -> int:
    return load().attn_prefill_varlen_window(q, kcache, vcache, o, lse, cu_seqlens_q, kv_lens, B, Hq,
                                             Hkv, total_q, max_sq, max_kv, d, int(window), int(n_sink),
                                             float(scale), o_dtype, stream)


def attn_decode_split(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale, n_splits,
                      min_rows_per_split, part_o, part_lse, stream) -> int:
    return load().attn_decode_split(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, float(scale),
                                    n_splits, min_rows_per_split, part_o, part_lse, stream)


def attn_merge(part_o, part_lse, o, lse, B, Hq, n_splits, d, o_dtype, stream) -> int:
    return load().attn_merge(part_o, part_lse, o, lse, B, Hq, n_splits, d, o_dtype, stream)


def attn_decode(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale, n_splits,
                min_rows_per_split, part_o, part_lse, o, lse, o_dtype, counters, stream) -> int:
    return load().attn_decode(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, float(scale),
                              n_splits, min_rows_per_split, part_o, part_lse, o, lse, o_dtype,
                              counters, stream)


def attn_prefill_schedule(BH, Sq, Skv, causal, grid, offsets, units, max_units) -> int:
    return load().attn_prefill_schedule(BH, Sq, Skv, int(causal), grid, offsets, units, max_units)


def prefill_schedule(BH: int, Sq: int, Skv: int, causal: bool, grid: int):
    """The causal prefill's unit lists, one per CTA (host only), or None when the
    launch deals its units in waves."""
    n_units = -(-Sq // 256) * BH
    offs = (ctypes.c_int * (grid + 1))()
    units = (ctypes.c_int * max(n_units, 1))()
    n = attn_prefill_schedule(BH, Sq, Skv, causal, grid, offs, units, n_units)
    if n < 0:
        raise AttnError(n, "attn_prefill_schedule")
    if n == 0:
        return None
    return [list(units[offs[c]:offs[c + 1]]) for c in range(grid)]


def attn_decode_noalloc(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv, scale, n_splits,
                        min_rows_per_split, o, lse, o_dtype, stream) -> int:
    return load().attn_decode_noalloc(q, kcache, vcache, kv_lens, B, Hq, Hkv, d, max_kv,
                                      float(scale), n_splits, min_rows_per_split, o, lse, o_dtype,
                                      stream)


def attn_decode_noalloc_scratch_bytes() -> int:
    return int(load().attn_decode_noalloc_scratch_bytes())


def attn_sync_check(stream) -> int:
    return load().attn_sync_check(stream)


def attn_strerror(status: int) -> str:
    return load().attn_strerror(int(status)).decode()


def attn_version() -> int:
    return load().attn_version()


def attn_debug_wait_timeout(limit_ns: int, stream) -> int:
    return load().attn_debug_wait_timeout(int(limit_ns), stream)


# ------------------------------------------------------------------ torch helpers
def _torch():
    import torch
    return torch


def _stream_handle(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_tensor(t, name, dtype, ndim):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _out_code(dtype):
    torch = _torch()
    if dtype == torch.float32:
        return ATTN_F32
    if dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported output dtype {dtype}")


def prefill(q, k, v, causal: bool = True, scale: float | None = None, out_dtype=None, stream=None,
            out=None, packed: bool = False):
    """Exact attention forward.  q [B,Sq,Hq,d], k/v [B,Skv,Hkv,d] bf16 on the GPU.
    packed=True folds the Hq/Hkv query heads of each KV head into the MMA tile rows
    (attn_prefill_packed).

    Returns (o [B,Sq,Hq,d] in out_dtype (default bf16), lse [B,Hq,Sq] fp32)."""
    torch = _torch()
    out_dtype = out_dtype or torch.bfloat16
    _check_tensor(q, "q", torch.bfloat16, 4)
    _check_tensor(k, "k", torch.bfloat16, 4)
    _check_tensor(v, "v", torch.bfloat16, 4)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        o = torch.empty((B, Sq, Hq, d), dtype=out_dtype, device=q.device)
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    fn = attn_prefill_packed if packed else attn_prefill_fwd
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv, d, causal, scale,
            _out_code(o.dtype), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, fn.__name__)
    return o, lse


def prefill_window(q, k, v, window: int, n_sink: int = 0, scale: float | None = None,
                   out_dtype=None, stream=None, out=None):
    """Causal prefill over a sliding window of ``window`` positions plus the first
    ``n_sink`` positions.  Shapes as ``prefill``; returns (o, lse)."""
    torch = _torch()
    out_dtype = out_dtype or torch.bfloat16
    _check_tensor(q, "q", torch.bfloat16, 4)
    _check_tensor(k, "k", torch.bfloat16, 4)
    _check_tensor(v, "v", torch.bfloat16, 4)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        o = torch.empty((B, Sq, Hq, d), dtype=out_dtype, device=q.device)
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    rc = attn_prefill_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv, d,
                             window, n_sink, scale, _out_code(o.dtype), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_prefill_window")
    return o, lse


def prefill_varlen(q, kcache, vcache, cu_seqlens_q, kv_lens, max_sq: int, causal: bool = True,
                   scale: float | None = None, out_dtype=None, stream=None, out=None,
                   window: int = 0, n_sink: int = 0):
    """Packed variable-length prefill against a KV cache (chunked prefill).

    q [total_q,Hq,d] bf16 (sequences concatenated), kcache/vcache [B,max_kv,Hkv,d] bf16,
    cu_seqlens_q int32 [B+1] and kv_lens int32 [B] on the GPU; max_sq >= the longest
    sequence.  window > 0 selects the causal sliding window of that many positions
    plus n_sink sink positions (attn_prefill_varlen_window; causal must be True).
    Returns (o [total_q,Hq,d] in out_dtype (default bf16), lse [Hq,total_q] fp32)."""
    torch = _torch()
    out_dtype = out_dtype or torch.bfloat16
    _check_tensor(q, "q", torch.bfloat16, 3)
    _check_tensor(kcache, "kcache", torch.bfloat16, 4)
    _check_tensor(vcache, "vcache", torch.bfloat16, 4)
    _check_tensor(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check_tensor(kv_lens, "kv_lens", torch.int32, 1)
    total_q, Hq, d = q.shape
    B, max_kv, Hkv, _ = kcache.shape
    if cu_seqlens_q.numel() != B + 1 or kv_lens.numel() != B:
        raise ValueError("cu_seqlens_q must have B+1 entries and kv_lens B")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        o = torch.empty((total_q, Hq, d), dtype=out_dtype, device=q.device)
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    if window:
        if not causal:
            raise ValueError("a sliding window is causal")
        rc = attn_prefill_varlen_window(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(o), _ptr(lse),
                                        _ptr(cu_seqlens_q), _ptr(kv_lens), B, Hq, Hkv, total_q,
                                        int(max_sq), max_kv, d, window, n_sink, scale,
                                        _out_code(o.dtype), _stream_handle(stream))
        if rc != ATTN_OK:
            raise AttnError(rc, "attn_prefill_varlen_window")
        return o, lse
    rc = attn_prefill_varlen(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(o), _ptr(lse),
                             _ptr(cu_seqlens_q), _ptr(kv_lens), B, Hq, Hkv, total_q, int(max_sq),
                             max_kv, d, causal, scale, _out_code(o.dtype), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_prefill_varlen")
    return o, lse


def decode_split(q, kcache, vcache, kv_lens, n_splits: int, min_rows_per_split: int = 1,
                 scale: float | None = None, stream=None, out=None):
    """Split-KV partials.  q [B,Hq,d], caches [B,max_kv,Hkv,d] bf16, kv_lens int32 [B].

    Returns (part_o [B,Hq,n_splits,d] fp32, part_lse [B,Hq,n_splits] fp32)."""
    torch = _torch()
    _check_tensor(q, "q", torch.bfloat16, 3)
    _check_tensor(kcache, "kcache", torch.bfloat16, 4)
    _check_tensor(vcache, "vcache", torch.bfloat16, 4)
    _check_tensor(kv_lens, "kv_lens", torch.int32, 1)
    B, Hq, d = q.shape
    _, max_kv, Hkv, _ = kcache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        part_o = torch.empty((B, Hq, n_splits, d), dtype=torch.float32, device=q.device)
        part_lse = torch.empty((B, Hq, n_splits), dtype=torch.float32, device=q.device)
    else:
        part_o, part_lse = out
    rc = attn_decode_split(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(kv_lens), B, Hq, Hkv, d, max_kv,
                           scale, n_splits, min_rows_per_split, _ptr(part_o), _ptr(part_lse),
                           _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_split")
    return part_o, part_lse


def merge(part_o, part_lse, out_dtype=None, stream=None, out=None):
    """LSE-weighted merge.  Returns (o [B,Hq,d] in out_dtype (default bf16), lse [B,Hq] fp32)."""
    torch = _torch()
    out_dtype = out_dtype or torch.bfloat16
    _check_tensor(part_o, "part_o", torch.float32, 4)
    _check_tensor(part_lse, "part_lse", torch.float32, 3)
    B, Hq, n_splits, d = part_o.shape
    if out is None:
        o = torch.empty((B, Hq, d), dtype=out_dtype, device=part_o.device)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=part_o.device)
    else:
        o, lse = out
    rc = attn_merge(_ptr(part_o), _ptr(part_lse), _ptr(o), _ptr(lse), B, Hq, n_splits, d,
                    _out_code(o.dtype), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_merge")
    return o, lse


_counters = {}  # (device type, index) -> the shared zeroed completion counters of decode()


def decode_counters(n: int, device):
    """The shared completion-counter buffer of decode() on `device`: int32, at least n
    entries, zero between calls.  Calls that use it must be ordered on one stream.
    It is allocated (and the device synchronised) when it first has to hold n
    entries: a call captured into a CUDA graph passes counters of its own, or
    follows a call of at least its size."""
    torch = _torch()
    key = (device.type, device.index)
    with _lock:
        buf = _counters.get(key)
        if buf is None or buf.numel() < n:
            buf = torch.zeros(max(n, 4096), dtype=torch.int32, device=device)
            torch.cuda.synchronize(device)  # zeroed before any stream uses it
            _counters[key] = buf
    return buf


def decode(q, kcache, vcache, kv_lens, n_splits: int, min_rows_per_split: int = 1,
           scale: float | None = None, out_dtype=None, stream=None, out=None, parts=None,
           counters=None):
    """Split-KV decode and its merge in one launch (attn_decode): (o [B,Hq,d], lse [B,Hq]).

    parts: optional (part_o [B,Hq,n_splits,d], part_lse [B,Hq,n_splits]) fp32 buffers for
    the split partials; counters: optional int32 [>= B*Hq] completion counters, zeroed by
    the caller (default: a buffer shared by the calls without their own)."""
    torch = _torch()
    _check_tensor(q, "q", torch.bfloat16, 3)
    _check_tensor(kcache, "kcache", torch.bfloat16, 4)
    _check_tensor(vcache, "vcache", torch.bfloat16, 4)
    _check_tensor(kv_lens, "kv_lens", torch.int32, 1)
    B, Hq, d = q.shape
    _, max_kv, Hkv, _ = kcache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if parts is None:
        part_o = torch.empty((B, Hq, n_splits, d), dtype=torch.float32, device=q.device)
        part_lse = torch.empty((B, Hq, n_splits), dtype=torch.float32, device=q.device)
    else:
        part_o, part_lse = parts
    if out is None:
        o = torch.empty((B, Hq, d), dtype=out_dtype or torch.bfloat16, device=q.device)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    if counters is None:
        counters = decode_counters(B * Hq, q.device)
    elif counters.dtype != torch.int32 or not counters.is_cuda or counters.numel() < B * Hq:
        raise TypeError("counters must be a CUDA int32 tensor of at least B*Hq entries")
    rc = attn_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(kv_lens), B, Hq, Hkv, d, max_kv,
                     scale, n_splits, min_rows_per_split, _ptr(part_o), _ptr(part_lse), _ptr(o),
                     _ptr(lse), _out_code(o.dtype), _ptr(counters), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode")
    return o, lse


def decode_split_packed(q, kcache, vcache, kv_lens, n_splits: int, min_rows_per_split: int = 1,
                        scale: float | None = None, stream=None, out=None):
    """Split-KV decode partials on the tensor cores (attn_decode_split_packed); same
    contract as decode_split.  Returns (part_o [B,Hq,n_splits,d], part_lse [B,Hq,n_splits])."""
    torch = _torch()
    _check_tensor(q, "q", torch.bfloat16, 3)
    _check_tensor(kcache, "kcache", torch.bfloat16, 4)
    _check_tensor(vcache, "vcache", torch.bfloat16, 4)
    _check_tensor(kv_lens, "kv_lens", torch.int32, 1)
    B, Hq, d = q.shape
    _, max_kv, Hkv, _ = kcache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        part_o = torch.empty((B, Hq, n_splits, d), dtype=torch.float32, device=q.device)
        part_lse = torch.empty((B, Hq, n_splits), dtype=torch.float32, device=q.device)
    else:
        part_o, part_lse = out
    rc = attn_decode_split_packed(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(kv_lens), B, Hq, Hkv, d,
                                  max_kv, scale, n_splits, min_rows_per_split, _ptr(part_o),
                                  _ptr(part_lse), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_split_packed")
    return part_o, part_lse


def decode_packed(q, kcache, vcache, kv_lens, scale: float | None = None, out_dtype=None,
                  stream=None, out=None, n_splits: int = 1, min_rows_per_split: int = 1):
    """One-token decode on the tensor cores, heads packed into the tile rows.
    q [B,Hq,d], caches [B,max_kv,Hkv,d] bf16, kv_lens int32 [B].  n_splits > 1 splits
    each sequence's keys (attn_decode_split_packed) and merges the partials
    (attn_merge); n_splits = 1 is one launch (attn_decode_packed).

    Returns (o [B,Hq,d] in out_dtype (default bf16), lse [B,Hq] fp32)."""
    if n_splits > 1:
        po, pl = decode_split_packed(q, kcache, vcache, kv_lens, n_splits, min_rows_per_split, scale,
                                     stream)
        return merge(po, pl, out_dtype, stream, out)
    torch = _torch()
    out_dtype = out_dtype or torch.bfloat16
    _check_tensor(q, "q", torch.bfloat16, 3)
    _check_tensor(kcache, "kcache", torch.bfloat16, 4)
    _check_tensor(vcache, "vcache", torch.bfloat16, 4)
    _check_tensor(kv_lens, "kv_lens", torch.int32, 1)
    B, Hq, d = q.shape
    _, max_kv, Hkv, _ = kcache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        o = torch.empty((B, Hq, d), dtype=out_dtype, device=q.device)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    rc = attn_decode_packed(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(kv_lens), B, Hq, Hkv, d, max_kv,
                            scale, _ptr(o), _ptr(lse), _out_code(o.dtype), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_packed")
    return o, lse


def sync_check(stream=None) -> None:
    """Synchronise `stream` and raise if a kernel recorded a device-side error.  After
    such an error the shared decode counters are zeroed again (their count is void)."""
    rc = attn_sync_check(_stream_handle(stream))
    if rc != ATTN_OK:
        with _lock:
            bufs = list(_counters.values())
        for buf in bufs:
            buf.zero_()
            _torch().cuda.synchronize(buf.device)
        raise AttnError(rc, "attn_sync_check")
