"""Causal sliding-window prefill with attention sinks, through the C ABI, against
the fp64 oracle.

Query i (key position p = i + Skv - Sq) admits the keys p - window < j <= p and
the sink keys j < n_sink (j <= p).  Small shapes are compared element by
element; the full-size windowed GQA prefill is compared on sampled rows that
the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_tcgen05_gb300 import prefill, prefill_window, sync_check
from attention_forward_tcgen05_gb300 import workloads as W
from tests.tolerances import check_lse, check_o

pytestmark = pytest.mark.gpu


def _inputs(B, Sq, Skv, Hq, Hkv, d, seed):
    s = W.PrefillShape("window_case", B, Hq, Hkv, Sq, Skv, d, True, 1.0 / np.sqrt(d), "f32", seed)
    return W.prefill_inputs_for(s)


def _run(q, k, v, window, n_sink, scale, out_dtype):
    o, lse = prefill_window(q.cuda(), k.cuda(), v.cuda(), window, n_sink, scale=scale, out_dtype=out_dtype)
    sync_check()
    return o.float().cpu().numpy(), lse.cpu().numpy()


# windows narrower than, equal to and wider than a KV tile, and one covering
# most keys; sink counts of none, part of a tile, a whole tile and several tiles
WINDOWS = [1, 64, 128, 200, 1000]
SINKS = [0, 4, 128, 300]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("n_sink", SINKS)
def test_window_sinks(d, window, n_sink):
    q, k, v = _inputs(1, 700, 700, 4, 2, d, 900 + d + window + n_sink)
    scale = 1.0 / np.sqrt(d)
    o, lse = _run(q, k, v, window, n_sink, scale, torch.float32)
    ro, rl = oracle.sdpa_window(q, k, v, window, n_sink, scale)
    check_o(o, ro, False)
    check_lse(lse, rl)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("Sq,Skv", [(300, 1100), (600, 257), (1, 513)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_window_unequal_lengths(d, Sq, Skv, out_dtype):
    """Queries at the end of a longer key sequence, and more queries than keys
    (the first rows then see no key at all)."""
    q, k, v = _inputs(2, Sq, Skv, 4, 1, d, 950 + d + Sq)
    scale = 0.7 / np.sqrt(d)
    o, lse = _run(q, k, v, 150, 20, scale, out_dtype)
    ro, rl = oracle.sdpa_window(q, k, v, 150, 20, scale)
    check_o(o, ro, out_dtype == torch.bfloat16)
    check_lse(lse, rl)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_window_covering_everything_equals_causal(d):
    """A window at least as long as the sequence admits every causal key: the
    result is the causal prefill's, bit for bit."""
    q, k, v = _inputs(1, 333, 333, 4, 4, d, 990 + d)
    o1, l1 = _run(q, k, v, 333, 0, 0.1, torch.float32)
    o2, l2 = _run(q, k, v, 5000, 17, 0.1, torch.float32)
    o3, l3 = prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=0.1, out_dtype=torch.float32)
    sync_check()
    np.testing.assert_array_equal(o1, o3.cpu().numpy())
    np.testing.assert_array_equal(l1, l3.cpu().numpy())
    np.testing.assert_array_equal(o2, o1)
    np.testing.assert_array_equal(l2, l1)


def test_no_keys():
    q, k, v = _inputs(1, 5, 0, 2, 2, 64, 997)
    o, lse = _run(q, k, v, 8, 2, 0.125, torch.float32)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
