"""Packed variable-length prefill against a KV cache (chunked prefill), through
the C ABI, against the fp64 oracle.

Small batches are compared element by element; the full-size chunked-prefill
workload is compared on sampled rows of every sequence that the oracle
computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_tcgen05_gb300 import prefill_varlen, sync_check
from attention_forward_tcgen05_gb300 import workloads as W
from tests.tolerances import check_lse, check_o

pytestmark = pytest.mark.gpu


def _run(q, kc, vc, cu, kv, causal, scale, out_dtype, max_sq=None):
    if max_sq is None:
        max_sq = int((cu[1:] - cu[:-1]).max().item()) if kv.numel() else 0
    o, lse = prefill_varlen(q.cuda(), kc.cuda(), vc.cuda(), cu.cuda(), kv.cuda(), max_sq,
                            causal=causal, scale=scale, out_dtype=out_dtype)
    sync_check()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _case(seqs, Hq, Hkv, d, seed, max_kv=None):
    sq = torch.tensor([a for a, _ in seqs], dtype=torch.int32)
    kv = torch.tensor([b for _, b in seqs], dtype=torch.int32)
    q, kc, vc, cu = W.varlen_inputs(len(seqs), Hq, Hkv, d, sq, kv, seed, max_kv)
    return q, kc, vc, cu, kv


# (new query rows, keys) per sequence: a single new token, a chunk after a
# history, a chunk that is the whole sequence, several KV tiles, an empty
# sequence, a sequence with fewer keys than rows (its first rows see no key
# under the causal mask), and a ragged tail in every dimension
MIXED = [(1, 1), (77, 300), (128, 128), (300, 1200), (0, 50), (200, 150), (129, 1000)]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_mixed_batch(d, causal, out_dtype):
    q, kc, vc, cu, kv = _case(MIXED, 4, 2, d, 60 + d)
    scale = 1.0 / np.sqrt(d)
    o, lse = _run(q, kc, vc, cu, kv, causal, scale, out_dtype)
    ro, rl = oracle.sdpa_varlen(q, kc, vc, cu, kv, causal, scale)
    check_o(o, ro, out_dtype == torch.bfloat16)
    check_lse(lse, rl)


def test_uneven_cached_prefixes():
    """Twenty sequences whose query chunks (1-599 rows) sit behind cached prefixes of
    up to 2,500 keys: a short chunk's one query block can outweigh every block of a
    long chunk with no history.  Every row against the oracle."""
    rng = np.random.default_rng(81)
    seqs = [(int(rng.integers(1, 600)), 0) for _ in range(20)]
    seqs = [(a, a + int(rng.integers(0, 2500))) for a, _ in seqs]
    q, kc, vc, cu, kv = _case(seqs, 4, 1, 64, 82)
    o, lse = _run(q, kc, vc, cu, kv, True, 0.125, torch.float32)
    ro, rl = oracle.sdpa_varlen(q, kc, vc, cu, kv, True, 0.125)
    check_o(o, ro, False)
    check_lse(lse, rl)


def test_many_short_sequences():
    """301 sequences, 300 of them a few rows long and one of 900 rows: 1,204
    (sequence, query block) units, most of them past their sequence's rows."""
    seqs = [(int(3 + (i * 7) % 20), int(3 + (i * 7) % 20 + (i * 13) % 90)) for i in range(300)] + [(900, 1000)]
    q, kc, vc, cu, kv = _case(seqs, 2, 1, 64, 83)
    o, lse = _run(q, kc, vc, cu, kv, True, 0.125, torch.float32)
    ro, rl = oracle.sdpa_varlen(q, kc, vc, cu, kv, True, 0.125)
    check_o(o, ro, False)
    check_lse(lse, rl)


def test_one_sequence_equals_prefill():
    """One sequence whose keys are exactly its rows is the fixed-length prefill."""
    from attention_forward_tcgen05_gb300 import prefill
    q, kc, vc, cu, kv = _case([(300, 300)], 8, 2, 128, 71)
    o1, l1 = _run(q, kc, vc, cu, kv, True, 0.1, torch.float32)
    o2, l2 = prefill(q[None].cuda(), kc.cuda(), vc.cuda(), causal=True, scale=0.1, out_dtype=torch.float32)
    sync_check()
    np.testing.assert_array_equal(o1, o2[0].cpu().numpy())
    np.testing.assert_array_equal(l1, l2[0].cpu().numpy())


def test_larger_max_sq_and_cache_than_needed():
    """max_sq and max_kv larger than every sequence: extra q-blocks do nothing and
    cache rows past kv_lens are never admitted (filled with large values here)."""
    q, kc, vc, cu, kv = _case([(90, 200), (33, 40)], 4, 4, 64, 72, max_kv=512)
    kc[:, 300:] = 30.0
    vc[:, 300:] = -30.0
    o, lse = _run(q, kc, vc, cu, kv, True, 0.125, torch.float32, max_sq=700)
    ro, rl = oracle.sdpa_varlen(q, kc, vc, cu, kv, True, 0.125)
    check_o(o, ro, False)
    check_lse(lse, rl)


def test_no_keys_anywhere():
    q, kc, vc, cu, kv = _case([(5, 0), (3, 0)], 2, 2, 64, 73, max_kv=0)
    o, lse = _run(q, kc, vc, cu, kv, True, 0.125, torch.float32)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


WINDOW_MIXED = [(200, 1500), (90, 90), (1, 700), (0, 64), (150, 100), (300, 600)]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("window,n_sink", [(1, 0), (100, 4), (256, 130), (2000, 7)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_mixed_batch_window(d, window, n_sink, out_dtype):
    q, kc, vc, cu, kv = _case(WINDOW_MIXED, 4, 2, d, 80 + d + window)
    scale = 1.0 / np.sqrt(d)
    max_sq = int((cu[1:] - cu[:-1]).max().item())
    o, lse = prefill_varlen(q.cuda(), kc.cuda(), vc.cuda(), cu.cuda(), kv.cuda(), max_sq, causal=True,
                            scale=scale, out_dtype=out_dtype, window=window, n_sink=n_sink)
    sync_check()
    ro, rl = oracle.sdpa_varlen_window(q, kc, vc, cu, kv, window, n_sink, scale)
    check_o(o.float().cpu().numpy(), ro, out_dtype == torch.bfloat16)
    check_lse(lse.cpu().numpy(), rl)
