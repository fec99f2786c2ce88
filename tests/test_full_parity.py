"""Every output element of the full-size workloads against the fp64 oracle.

Each workload runs through the public API in the launch configuration the
benchmark times (same shapes, split policies and output types), and the whole
output -- every O element and every LSE -- is compared with the oracle's, at
the tolerances of ``tests/tolerances.py``.  The prefill workloads run with
both output types: fp32 O shows the kernel's arithmetic error alone, bf16 O
adds the output's own rounding.  The oracle of a workload is computed once and
shared by its tests.  The largest errors are printed at the end of the session.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from attention_forward_tcgen05_gb300 import (decode, decode_packed, prefill, prefill_varlen, prefill_window,
                                             sync_check)
from attention_forward_tcgen05_gb300 import workloads as W
from tests.tolerances import check_lse, check_o, log_parity

pytestmark = pytest.mark.gpu

DTYPES = [torch.bfloat16, torch.float32]
DT_IDS = ["o_bf16", "o_f32"]


def _compare(what, o, lse, ro, rl, out_dtype):
    got_o = o.float().cpu().numpy()
    got_l = lse.cpu().numpy()
    eo = check_o(got_o, ro, out_dtype == torch.bfloat16, f"{what} O")
    el = check_lse(got_l, rl, f"{what} LSE")
    log_parity(what, eo, el)


# ---------------------------------------------------------------- fixed-length prefill
PREFILL_SHAPES = {s.name: s for s in (W.GQA_PREFILL, W.mha_sweep(64), W.mha_sweep(128), W.mha_sweep(256),
                                       W.mha_sweep(512))}


@functools.lru_cache(maxsize=None)
def _prefill_case(name):
    s = PREFILL_SHAPES[name]
    q, k, v = W.prefill_inputs_for(s)
    ro, rl = oracle.sdpa(q, k, v, s.causal, s.scale)
    return s, (q, k, v), ro, rl


@pytest.mark.parametrize("name", list(PREFILL_SHAPES))
@pytest.mark.parametrize("out_dtype", DTYPES, ids=DT_IDS)
def test_prefill_workload_whole_output(name, out_dtype):
    """The causal GQA prefill (S = 3314) and the non-causal head-dim sweep
    (S = 4096, d = 64, 128, 256, and 512): every row of every head."""
    s, (q, k, v), ro, rl = _prefill_case(name)
    o, lse = prefill(q.cuda(), k.cuda(), v.cuda(), causal=s.causal, scale=s.scale, out_dtype=out_dtype)
    sync_check()
    _compare(f"{s.name} ({DT_IDS[DTYPES.index(out_dtype)]})", o, lse, ro, rl, out_dtype)


# ---------------------------------------------------------------- sliding window + sinks
@functools.lru_cache(maxsize=1)
def _window_case():
    s = W.WINDOW_PREFILL
    q, k, v = W.prefill_inputs_for(s.base)
    ro, rl = oracle.sdpa_window(q, k, v, s.window, s.n_sink, s.base.scale)
    return s, (q, k, v), ro, rl


@pytest.mark.parametrize("out_dtype", DTYPES, ids=DT_IDS)
def test_window_workload_whole_output(out_dtype):
    s, (q, k, v), ro, rl = _window_case()
    o, lse = prefill_window(q.cuda(), k.cuda(), v.cuda(), s.window, s.n_sink, scale=s.base.scale,
                            out_dtype=out_dtype)
    sync_check()
    _compare(f"{s.name} ({DT_IDS[DTYPES.index(out_dtype)]})", o, lse, ro, rl, out_dtype)


# ---------------------------------------------------------------- chunked (varlen) prefill
@functools.lru_cache(maxsize=1)
def _chunked_case():
    s = W.CHUNKED_PREFILL
    q, kc, vc, cu, kv = W.varlen_inputs_for(s)
    ro, rl = oracle.sdpa_varlen(q, kc, vc, cu, kv, s.causal, s.scale)
    return s, (q, kc, vc, cu, kv), ro, rl


@pytest.mark.parametrize("out_dtype", DTYPES, ids=DT_IDS)
def test_chunked_prefill_workload_whole_output(out_dtype):
    s, (q, kc, vc, cu, kv), ro, rl = _chunked_case()
    max_sq = int((cu[1:] - cu[:-1]).max())
    o, lse = prefill_varlen(q.cuda(), kc.cuda(), vc.cuda(), cu.cuda(), kv.cuda(), max_sq, causal=s.causal,
                            scale=s.scale, out_dtype=out_dtype)
    sync_check()
    _compare(f"{s.name} ({DT_IDS[DTYPES.index(out_dtype)]})", o, lse, ro, rl, out_dtype)


# ---------------------------------------------------------------- decode
@functools.lru_cache(maxsize=None)
def _decode_case(name):
    s = {W.GQA_DECODE.name: W.GQA_DECODE, W.RAGGED_DECODE.name: W.RAGGED_DECODE,
         W.MQA_DECODE.name: W.MQA_DECODE}[name]
    q, kc, vc, lens = W.decode_inputs_for(s)
    ro, rl = oracle.decode(q, kc, vc, lens, s.scale)
    return s, (q, kc, vc, lens), ro, rl


@pytest.mark.parametrize("name", [W.GQA_DECODE.name, W.RAGGED_DECODE.name])
def test_split_decode_workload_whole_output(name):
    """Split-KV decode + merge (CUDA cores) with the benchmark's split policy,
    bf16 O: every head of every sequence."""
    s, (q, kc, vc, lens), ro, rl = _decode_case(name)
    o, lse = decode(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), s.n_splits, s.min_rows_per_split, s.scale,
                    torch.bfloat16)
    sync_check()
    _compare(f"{s.name} (split + merge, o_bf16)", o, lse, ro, rl, torch.bfloat16)


@pytest.mark.parametrize("splits", [None, W.MQA_DECODE_SPLITS], ids=["one_launch", "split_merge"])
def test_mqa_decode_workload_whole_output(splits):
    """The 128-head multi-query decode on the tensor cores (all 128 sequences),
    in one launch as the benchmark runs it, and through split partials + merge."""
    s, (q, kc, vc, lens), ro, rl = _decode_case(W.MQA_DECODE.name)
    kw = {} if splits is None else {"n_splits": splits[0], "min_rows_per_split": splits[1]}
    o, lse = decode_packed(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), s.scale, **kw)
    sync_check()
    _compare(f"{s.name} ({'one launch' if splits is None else 'split + merge'}, o_bf16)", o, lse, ro, rl,
             torch.bfloat16)
