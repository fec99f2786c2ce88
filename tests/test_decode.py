"""Split-KV decode and merge against the fp64 oracle, through the C ABI; the decode with
the combine fused into the split launch against the two launches."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_tcgen05_gb300 as attn
from attention_forward_tcgen05_gb300 import decode, decode_split, merge, sync_check
from attention_forward_tcgen05_gb300 import workloads as W
from tests.tolerances import check_lse, check_o

pytestmark = pytest.mark.gpu


def _fused(args, n_splits, min_rows, scale, out_dtype, o, lse, po, pl):
    """attn_decode (the combine in the split launch) on the same inputs: its partials,
    O and LSE are bit-identical to the two launches (the same arithmetic), and every
    group's completion counter is back at zero afterwards."""
    B, Hq = args[0].shape[0], args[0].shape[1]
    ctr = torch.zeros(B * Hq, dtype=torch.int32, device="cuda")
    fpo, fpl = torch.full_like(po, float("nan")), torch.full_like(pl, float("nan"))
    fo, fl = decode(*args, n_splits, min_rows, scale, out_dtype, parts=(fpo, fpl), counters=ctr)
    sync_check()
    assert torch.equal(fpo, po) and torch.equal(fpl, pl), "fused decode partials differ"
    assert torch.equal(fo, o) and torch.equal(fl, lse), "fused decode O / LSE differ from split + merge"
    assert not torch.any(ctr).item(), "completion counters not reset"


def _compare(q, kc, vc, lens, n_splits, min_rows, scale, out_dtype=torch.bfloat16):
    args = (q.cuda(), kc.cuda(), vc.cuda(), lens.cuda())
    po, pl = decode_split(*args, n_splits, min_rows, scale)
    o, lse = merge(po, pl, out_dtype)
    sync_check()  # a bounded pipeline wait that ran out would surface here
    _fused(args, n_splits, min_rows, scale, out_dtype, o, lse, po, pl)
    rpo, rpl = oracle.decode_split(q, kc, vc, lens, scale, n_splits, min_rows)
    ro, rl = oracle.decode(q, kc, vc, lens, scale)
    check_lse(pl.cpu().numpy(), rpl, "part_lse")
    check_o(po.cpu().numpy(), rpo, False, "part_o")
    check_o(o.float().cpu().numpy(), ro, out_dtype == torch.bfloat16, "O")
    check_lse(lse.cpu().numpy(), rl, "LSE")


def test_gqa_decode_1641():
    s = W.GQA_DECODE
    q, kc, vc, lens = W.decode_inputs_for(s)
    _compare(q, kc, vc, lens, s.n_splits, s.min_rows_per_split, s.scale)


@pytest.mark.parametrize("n_splits,min_rows", [(1, 1), (8, 1), (16, 64), (3, 0)])
def test_nkv_edges(n_splits, min_rows):
    lens = torch.tensor([1, 29, 52, 512, 1641, 0], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(6, 28, 4, 128, lens, 321)
    _compare(q, kc, vc, lens, n_splits, min_rows, 1.0 / math.sqrt(128))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (10, 2), (16, 2), (32, 2), (34, 2), (56, 2), (128, 1)])
def test_head_ratios_and_dims(d, Hq, Hkv):
    """Groups of 1 to 128 query heads per KV head: above 16 heads a group is always
    spread over several CTAs (here, a small launch, it is spread further still)."""
    lens = torch.tensor([33, 700, 95], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(3, Hq, Hkv, d, lens, 17 + d + Hq, Lmax=720)
    _compare(q, kc, vc, lens, 4, 16, 1.0 / math.sqrt(d), torch.float32)


@pytest.mark.parametrize("Hq,Hkv,n_splits", [(34, 2, 2), (128, 1, 4)])
def test_large_groups_many_units(Hq, Hkv, n_splits):
    """A launch of at least 128 (sequence, KV head, split) units whose group is above
    16 heads: the group is split only as far as the per-CTA limit needs (17 -> 9 + 8,
    128 -> 8 x 16), with an empty sequence and splits of one row."""
    g = torch.Generator().manual_seed(Hq)
    lens = torch.randint(1, 300, (40,), generator=g, dtype=torch.int32)
    lens[:3] = torch.tensor([0, 1, 2], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(40, Hq, Hkv, 128, lens, 600 + Hq, Lmax=300)
    _compare(q, kc, vc, lens, n_splits, 1, 1.0 / math.sqrt(128))


def test_large_scores():
    lens = torch.tensor([900, 64], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(2, 8, 2, 128, lens, 5)
    q = (q.float() * 4).to(torch.bfloat16)
    _compare(q, kc, vc, lens, 5, 1, 0.5)


@pytest.mark.parametrize("policy", ["workload", "8x1024"])
def test_ragged_b64_full(policy):
    # the benchmark's split policy, and 8 splits of at least 1024 rows
    s = W.RAGGED_DECODE
    q, kc, vc, lens = W.decode_inputs_for(s)
    ns, mr = (s.n_splits, s.min_rows_per_split) if policy == "workload" else (8, 1024)
    _compare(q, kc, vc, lens, ns, mr, s.scale)


def test_ragged_b64_sixteen_splits():
    # the same batch split finer: 16 splits of at least 512 rows, so short
    # sequences leave up to 15 empty splits that the merge must skip
    s = W.RAGGED_DECODE
    q, kc, vc, lens = W.decode_inputs_for(s)
    _compare(q, kc, vc, lens, 16, 512, s.scale)


def test_merge_random_partials():
    rng = np.random.default_rng(2)
    B, Hq, S, d = 3, 5, 7, 128
    po = torch.from_numpy(rng.standard_normal((B, Hq, S, d)).astype(np.float32))
    pl = torch.from_numpy((rng.standard_normal((B, Hq, S)) * 4).astype(np.float32))
    pl[0, 1, 2:] = -math.inf
    pl[1, 3, :] = -math.inf          # every split empty: O = 0, LSE = -inf
    po[pl == -math.inf] = 0.0
    o, lse = merge(po.cuda(), pl.cuda(), torch.float32)
    torch.cuda.synchronize()
    ro, rl = oracle.merge(po, pl)
    check_o(o.cpu().numpy(), ro, False)
    check_lse(lse.cpu().numpy(), rl)


def _order_lens(B, hi, seed, edges):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(0, hi + 1, (B,), generator=g, dtype=torch.int32)
    lens[: len(edges)] = torch.tensor(edges, dtype=torch.int32)
    return lens


@pytest.mark.parametrize("n_splits,min_rows", [(8, 64), (5, 1)])
def test_unit_order_ragged_tails(n_splits, min_rows):
    """The launch runs full splits first, then the partial last splits by size,
    then the empty ones.  Lengths cover every size bucket of the partial splits,
    ties inside a bucket, sequences with no partial split (multiples of the
    chunk), empty sequences, and a batch that is not a multiple of 32."""
    edges = [0, 64, 128, 512, 1, 3, 4, 63, 65, 100, 127, 129, 191, 255, 256, 257, 511, 513, 0, 4, 4, 1500]
    lens = _order_lens(70, 1500, 77 + n_splits, edges)
    q, kc, vc = W.decode_inputs(70, 8, 2, 128, lens, 78 + n_splits, Lmax=1500)
    _compare(q, kc, vc, lens, n_splits, min_rows, 1.0 / math.sqrt(128))


@pytest.mark.parametrize("B", [1024, 1030])
def test_unit_order_large_batches(B):
    """1024 sequences: the largest batch that takes the size order (32 passes of
    the warp over the lengths); 1030 takes the batch-major order."""
    lens = _order_lens(B, 40, B, [0, 1, 8, 16, 40])
    q, kc, vc = W.decode_inputs(B, 4, 2, 64, lens, B + 1, Lmax=40)
    _compare(q, kc, vc, lens, 4, 8, 0.125, torch.float32)


def test_unit_order_no_partial_splits():
    """Every length a multiple of its chunk (8 splits, at least 64 rows each):
    the launch has full and empty units only."""
    lens = torch.tensor([64, 128, 512, 1024, 0, 192, 2048, 64, 448, 320], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(10, 8, 2, 128, lens, 91, Lmax=2048)
    _compare(q, kc, vc, lens, 8, 64, 1.0 / math.sqrt(128))


def test_unit_order_all_empty():
    """No sequence has keys: every unit is empty, O = 0 and LSE = -inf."""
    lens = torch.zeros(40, dtype=torch.int32)
    q, kc, vc = W.decode_inputs(40, 8, 2, 64, lens, 92, Lmax=16)
    args = (q.cuda(), kc.cuda(), vc.cuda(), lens.cuda())
    po, pl = decode_split(*args, 8, 1, 0.125)
    o, lse = merge(po, pl, torch.float32)
    sync_check()
    assert torch.all(pl.cpu() == -math.inf) and torch.all(po.cpu() == 0)
    assert torch.all(o.cpu() == 0) and torch.all(lse.cpu() == -math.inf)
    _fused(args, 8, 1, 0.125, torch.float32, o, lse, po, pl)


def test_fused_decode_shared_counters():
    """decode() without counters of its own uses the binding's shared buffer: calls of
    different shapes and split counts in sequence each see zeroed counters, and the
    buffer is zero again after them."""
    cases = [([1641, 0, 7, 300], 28, 4, 128, 8, 1), ([50, 2048], 32, 8, 64, 16, 64),
             ([1641], 28, 4, 128, 8, 1), ([5, 0, 0], 8, 2, 256, 3, 0)]
    for i, (lens, Hq, Hkv, d, ns, mr) in enumerate(cases):
        lens = torch.tensor(lens, dtype=torch.int32)
        q, kc, vc = W.decode_inputs(len(lens), Hq, Hkv, d, lens, 500 + i)
        scale = 1.0 / math.sqrt(d)
        o, lse = decode(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), ns, mr, scale, torch.float32)
        sync_check()
        ro, rl = oracle.decode(q, kc, vc, lens, scale)
        check_o(o.cpu().numpy(), ro, False, f"case {i} O")
        check_lse(lse.cpu().numpy(), rl, f"case {i} LSE")
    assert not torch.any(attn.decode_counters(1, torch.device("cuda", torch.cuda.current_device()))).item()


def test_max_splits():
    """The largest split count (1024) on short sequences: most units hold one or
    two rows or none, and the merge walks 32 batches of split weights."""
    lens = torch.tensor([1500, 1, 700], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(3, 8, 2, 128, lens, 93, Lmax=1500)
    _compare(q, kc, vc, lens, 1024, 1, 1.0 / math.sqrt(128))
