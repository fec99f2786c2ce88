"""attn_decode_noalloc: split-KV decode + merge without any device allocation.

Callers that cannot call cudaMalloc (a memory pool that already reserved the
device, code that must not synchronise the device, C callers without a device
allocator) use this entry point; its split partials live in the library's
static device array.  The test calls it through the C ABI and compares with
attn_decode_split + attn_merge on caller-allocated partials, and with the
fp64 oracle's decode, within the parity tolerances, on two calls in a row --
the second one smaller, so stale contents of the shared array from the first
call must not leak into it.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import attention_forward_tcgen05_gb300 as attn
import oracle
from attention_forward_tcgen05_gb300 import workloads as W
from tests.tolerances import check_lse, check_o

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(q, kc, vc, lens, n_splits, min_rows, scale, out_dtype):
    B, Hq, d = q.shape
    _, max_kv, Hkv, _ = kc.shape
    o = torch.empty((B, Hq, d), dtype=out_dtype, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    code = attn.ATTN_BF16 if out_dtype == torch.bfloat16 else attn.ATTN_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = attn.attn_decode_noalloc(_p(q), _p(kc), _p(vc), _p(lens), B, Hq, Hkv, d, max_kv, scale,
                                  n_splits, min_rows, _p(o), _p(lse), code, stream)
    assert rc == attn.ATTN_OK, attn.attn_strerror(rc)
    return o, lse


def _case(lens, Hq, Hkv, d, seed):
    lens = torch.tensor(lens, dtype=torch.int32)
    q, kc, vc = W.decode_inputs(len(lens), Hq, Hkv, d, lens, seed)
    return (q, kc, vc, lens), (q.cuda(), kc.cuda(), vc.cuda(), lens.cuda())


def test_noalloc_matches_decode_split_and_merge_twice():
    calls = [
        # (lens, Hq, Hkv, d, n_splits, min_rows, out dtype) -- the first call fills more of the
        # shared array than the second one reads
        ([1641, 29, 0, 512, 3000, 77], 28, 4, 128, 16, 1, torch.bfloat16),
        ([300, 5], 8, 2, 64, 4, 0, torch.float32),
    ]
    for i, (lens, Hq, Hkv, d, n_splits, min_rows, odt) in enumerate(calls):
        host, (q, kc, vc, lg) = _case(lens, Hq, Hkv, d, 100 + i)
        scale = 1.0 / math.sqrt(d)
        o_ref, l_ref = attn.decode(q, kc, vc, lg, n_splits, min_rows, scale, odt)
        o, l = _noalloc(q, kc, vc, lg, n_splits, min_rows, scale, odt)
        assert attn.attn_sync_check(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
        got_o, got_l = o.float().cpu().numpy(), l.cpu().numpy()
        # against the entry point that takes caller-allocated partials ...
        check_o(got_o, o_ref.float().cpu().numpy(), odt == torch.bfloat16, f"call {i} O vs decode")
        check_lse(got_l, l_ref.cpu().numpy(), f"call {i} LSE vs decode")
        # ... and against the fp64 oracle's unsplit decode
        ro, rl = oracle.decode(*host, scale)
        check_o(got_o, ro, odt == torch.bfloat16, f"call {i} O vs oracle")
        check_lse(got_l, rl, f"call {i} LSE vs oracle")
