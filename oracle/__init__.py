"""fp64 CPU oracle for exact scaled-dot-product attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  It shares no code with the CUDA
library and never calls it.  The arithmetic lives in ``attn_oracle.c``
(plain C, fp64); this module only marshals numpy arrays through ctypes.

Inputs may be numpy arrays or torch tensors of any float dtype; they are
widened to fp64 exactly (bf16 -> fp64 is exact).  Layouts are the ones the
C file states: prefill q/o ``[B, Sq, Hq, d]``, k/v ``[B, Skv, Hkv, d]``,
lse ``[B, Hq, Sq]``; decode q/o ``[B, Hq, d]``, caches ``[B, Lmax, Hkv, d]``,
part_o ``[B, Hq, n_splits, d]``, part_lse ``[B, Hq, n_splits]``; packed
variable-length prefill q/o ``[total_q, Hq, d]``, lse ``[Hq, total_q]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle C source to a shared library with gcc (-O2, plain C99,
    no ISA-specific flags, so it builds the same on x86-64 and aarch64)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", "-o", tmp, src,
             "-lm", "-lpthread"])
        os.replace(tmp, out)
    return out


def _bind(lib):
    P = ctypes.POINTER(ctypes.c_double)
    I = ctypes.POINTER(ctypes.c_int)
    c_int, c_double = ctypes.c_int, ctypes.c_double
    lib.oracle_sdpa.argtypes = [P, P, P] + [c_int] * 7 + [c_double, P, P, c_int]
    lib.oracle_sdpa_rows.argtypes = [P, P, P] + [c_int] * 7 + [c_double, I, c_int, P, P, c_int]
    lib.oracle_sdpa_window.argtypes = [P, P, P] + [c_int] * 8 + [c_double, P, P, c_int]
    lib.oracle_sdpa_window_rows.argtypes = [P, P, P] + [c_int] * 8 + [c_double, I, c_int, P, P, c_int]
    lib.oracle_split_bounds.argtypes = [c_int] * 4 + [I, I]
    lib.oracle_decode_split.argtypes = [P, P, P, I] + [c_int] * 5 + [c_double, c_int, c_int, P, P, c_int]
    lib.oracle_decode.argtypes = [P, P, P, I] + [c_int] * 5 + [c_double, P, P, c_int]
    lib.oracle_merge.argtypes = [P, P] + [c_int] * 4 + [P, P]
    lib.oracle_num_cores.argtypes = []
    for f in ("oracle_sdpa", "oracle_sdpa_rows", "oracle_split_bounds", "oracle_decode_split",
              "oracle_decode", "oracle_merge", "oracle_num_cores", "oracle_sdpa_window",
              "oracle_sdpa_window_rows"):
        getattr(lib, f).restype = c_int
    return lib


_default = None


def _load():
    global _default
    with _lock:
        if _default is None:
            _default = _bind(ctypes.CDLL(build()))
    return _default


def load_variant(path: str):
    """Load another build of the oracle source (used by the tests that plant a
    mistake in a copy of the oracle and check that a pin catches it)."""
    return _bind(ctypes.CDLL(path))


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what} failed with oracle status {rc}")


def num_cores(lib=None) -> int:
    return int((lib or _load()).oracle_num_cores())


def sdpa(q, k, v, causal: bool, scale: float, nthreads: int = 0, lib=None):
    """Exact attention, prefill shape.  Returns (o [B,Sq,Hq,d], lse [B,Hq,Sq]) in fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    o = np.zeros((B, Sq, Hq, d), np.float64)
    lse = np.zeros((B, Hq, Sq), np.float64)
    rc = (lib or _load()).oracle_sdpa(_dp(q), _dp(k), _dp(v), B, Hq, Hkv, Sq, Skv, d, int(bool(causal)),
                             float(scale), _dp(o), _dp(lse), int(nthreads))
    _check(rc, "oracle_sdpa")
    return o, lse


def sdpa_window(q, k, v, window: int, n_sink: int, scale: float, nthreads: int = 0, lib=None):
    """Causal attention over a sliding window plus attention sinks: query i (key
    position p = i + Skv - Sq) admits the keys p - window < j <= p and the first
    n_sink keys j < n_sink (j <= p).  Same layouts as ``sdpa``.  Follows the
    sliding-window and sink items (D3-D5) of "STAGE_D.md -- FMHA Kernel
    Development": their two branches merged through the LSE are exactly the
    softmax over the union of the two key sets, which this computes directly."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    o = np.zeros((B, Sq, Hq, d), np.float64)
    lse = np.zeros((B, Hq, Sq), np.float64)
    rc = (lib or _load()).oracle_sdpa_window(_dp(q), _dp(k), _dp(v), B, Hq, Hkv, Sq, Skv, d, int(window),
                                             int(n_sink), float(scale), _dp(o), _dp(lse), int(nthreads))
    _check(rc, "oracle_sdpa_window")
    return o, lse


def sdpa_window_rows(q, k, v, window: int, n_sink: int, scale: float, rows, nthreads: int = 0, lib=None):
    """Selected rows ``rows`` = [(b, hq, i), ...] of ``sdpa_window``: (o [n, d], lse [n])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    r = _i32(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = r.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = (lib or _load()).oracle_sdpa_window_rows(_dp(q), _dp(k), _dp(v), B, Hq, Hkv, Sq, Skv, d, int(window),
                                                  int(n_sink), float(scale), _ip(r), n, _dp(o), _dp(lse),
                                                  int(nthreads))
    _check(rc, "oracle_sdpa_window_rows")
    return o, lse


def sdpa_varlen(q, kcache, vcache, cu_seqlens_q, kv_lens, causal: bool, scale: float,
                nthreads: int = 0, lib=None):
    """Packed variable-length prefill against a KV cache, by its definition: every
    sequence b is the plain prefill of its own rows q[cu[b]:cu[b+1]] against the
    keys kcache[b, :kv_lens[b]] (bottom-right causal alignment when Sq_b < L_b:
    the new rows are the sequence's last positions), computed with ``sdpa``.
    Layouts: q/o ``[total_q, Hq, d]``, caches ``[B, max_kv, Hkv, d]``, lse ``[Hq, total_q]``.
    Follows the per-sequence key bound of "60 . r57 -- FA KV staging double
    buffering (REVERTED)", section 2.2; the per-sequence computation is ``sdpa``."""
    q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
    cu = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    lens = [int(x) for x in np.asarray(kv_lens).reshape(-1)]
    total_q, Hq, d = q.shape
    o = np.zeros((total_q, Hq, d), np.float64)
    lse = np.full((Hq, total_q), -np.inf, np.float64)
    for b, L in enumerate(lens):
        c0, c1 = cu[b], cu[b + 1]
        if c1 <= c0:
            continue
        ob, lb = sdpa(q[None, c0:c1], kc[b:b + 1, :L], vc[b:b + 1, :L], causal, scale, nthreads, lib)
        o[c0:c1] = ob[0]
        lse[:, c0:c1] = lb[0]
    return o, lse


def sdpa_varlen_window(q, kcache, vcache, cu_seqlens_q, kv_lens, window: int, n_sink: int,
                       scale: float, nthreads: int = 0, lib=None):
    """Packed variable-length causal prefill over a sliding window plus sinks:
    every sequence b is ``sdpa_window`` of its own rows q[cu[b]:cu[b+1]] against the
    keys kcache[b, :kv_lens[b]].  Layouts as ``sdpa_varlen``.  kv_lens is the
    per-sequence window length of the sliding-window items (D3) of "STAGE_D.md --
    FMHA Kernel Development"; the per-sequence computation is ``sdpa_window``."""
    q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
    cu = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    lens = [int(x) for x in np.asarray(kv_lens).reshape(-1)]
    total_q, Hq, d = q.shape
    o = np.zeros((total_q, Hq, d), np.float64)
    lse = np.full((Hq, total_q), -np.inf, np.float64)
    for b, L in enumerate(lens):
        c0, c1 = cu[b], cu[b + 1]
        if c1 <= c0:
            continue
        ob, lb = sdpa_window(q[None, c0:c1], kc[b:b + 1, :L], vc[b:b + 1, :L], window, n_sink, scale,
                             nthreads, lib)
        o[c0:c1] = ob[0]
        lse[:, c0:c1] = lb[0]
    return o, lse


def sdpa_rows(q, k, v, causal: bool, scale: float, rows, nthreads: int = 0, lib=None):
    """Exact attention for selected rows ``rows`` = [(b, hq, i), ...].

    Returns (o [n, d], lse [n]) in fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    r = _i32(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = r.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = (lib or _load()).oracle_sdpa_rows(_dp(q), _dp(k), _dp(v), B, Hq, Hkv, Sq, Skv, d, int(bool(causal)),
                                  float(scale), _ip(r), n, _dp(o), _dp(lse), int(nthreads))
    _check(rc, "oracle_sdpa_rows")
    return o, lse


def split_bounds(L: int, n_splits: int, min_rows: int, s: int, lib=None):
    lo, hi = ctypes.c_int(0), ctypes.c_int(0)
    rc = (lib or _load()).oracle_split_bounds(int(L), int(n_splits), int(min_rows), int(s),
                                     ctypes.byref(lo), ctypes.byref(hi))
    _check(rc, "oracle_split_bounds")
    return lo.value, hi.value


def decode_split(q, kc, vc, kv_lens, scale: float, n_splits: int, min_rows: int, nthreads: int = 0, lib=None):
    """Per-split partials.  Returns (part_o [B,Hq,n_splits,d], part_lse [B,Hq,n_splits])."""
    q, kc, vc, lens = _f64(q), _f64(kc), _f64(vc), _i32(kv_lens)
    B, Hq, d = q.shape
    _, Lmax, Hkv, _ = kc.shape
    po = np.zeros((B, Hq, n_splits, d), np.float64)
    pl = np.zeros((B, Hq, n_splits), np.float64)
    rc = (lib or _load()).oracle_decode_split(_dp(q), _dp(kc), _dp(vc), _ip(lens), B, Hq, Hkv, d, Lmax,
                                     float(scale), int(n_splits), int(min_rows), _dp(po), _dp(pl),
                                     int(nthreads))
    _check(rc, "oracle_decode_split")
    return po, pl


def decode(q, kc, vc, kv_lens, scale: float, nthreads: int = 0, lib=None):
    """Unsplit decode.  Returns (o [B,Hq,d], lse [B,Hq])."""
    q, kc, vc, lens = _f64(q), _f64(kc), _f64(vc), _i32(kv_lens)
    B, Hq, d = q.shape
    _, Lmax, Hkv, _ = kc.shape
    o = np.zeros((B, Hq, d), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = (lib or _load()).oracle_decode(_dp(q), _dp(kc), _dp(vc), _ip(lens), B, Hq, Hkv, d, Lmax,
                               float(scale), _dp(o), _dp(lse), int(nthreads))
    _check(rc, "oracle_decode")
    return o, lse


def merge(part_o, part_lse, lib=None):
    """LSE-weighted merge.  Returns (o [B,Hq,d], lse [B,Hq])."""
    po, pl = _f64(part_o), _f64(part_lse)
    B, Hq, n_splits, d = po.shape
    o = np.zeros((B, Hq, d), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = (lib or _load()).oracle_merge(_dp(po), _dp(pl), B, Hq, n_splits, d, _dp(o), _dp(lse))
    _check(rc, "oracle_merge")
    return o, lse
