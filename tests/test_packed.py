"""Head packing (the query heads of one KV head folded into the MMA tile rows),
through the C ABI: attn_prefill_packed against the fp64 oracle and bit for bit
against the unpacked kernel, attn_decode_packed against the oracle's decode.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_tcgen05_gb300 import decode_packed, prefill, sync_check
from attention_forward_tcgen05_gb300 import workloads as W
from tests.tolerances import check_lse, check_o

pytestmark = pytest.mark.gpu


def _prefill_inputs(B, Sq, Skv, Hq, Hkv, d, seed):
    s = W.PrefillShape("packed_case", B, Hq, Hkv, Sq, Skv, d, True, 1.0 / np.sqrt(d), "f32", seed)
    return W.prefill_inputs_for(s)


# (Hq, Hkv): MQA groups of 2..128 heads and a GQA group of 8
GROUPS = [(128, 1), (16, 1), (2, 1), (32, 4), (8, 4)]
# (Sq, Skv): single token, a few positions (a tile holds 128/G of them), a ragged
# tail across several tiles, more keys than queries, more queries than keys
LENGTHS = [(1, 300), (5, 5), (77, 640), (300, 300), (40, 23)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", GROUPS)
@pytest.mark.parametrize("Sq,Skv", LENGTHS)
@pytest.mark.parametrize("causal", [True, False])
def test_packed_prefill(d, Hq, Hkv, Sq, Skv, causal):
    q, k, v = _prefill_inputs(2, Sq, Skv, Hq, Hkv, d, 500 + d + Hq + Sq)
    scale = 1.0 / np.sqrt(d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = prefill(qd, kd, vd, causal=causal, scale=scale, out_dtype=torch.float32, packed=True)
    o2, lse2 = prefill(qd, kd, vd, causal=causal, scale=scale, out_dtype=torch.float32)
    sync_check()
    o, lse = o.cpu().numpy(), lse.cpu().numpy()
    # the same rows, keys, masks and per-row arithmetic as the unpacked kernel --
    # unless the unpacked launch ran its last wave as key halves (a non-causal
    # launch over more units than SMs with a last wave at most half full)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    units = -(-Sq // 256) * Hq * 2
    halves_tail = (not causal) and units > n_sm and 0 < units % n_sm <= n_sm // 2
    if not halves_tail:
        np.testing.assert_array_equal(o, o2.cpu().numpy())
        np.testing.assert_array_equal(lse, lse2.cpu().numpy())
    ro, rl = oracle.sdpa(q, k, v, causal, scale)
    check_o(o, ro, False)
    check_lse(lse, rl)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_packed_prefill_bf16_output(out_dtype):
    q, k, v = _prefill_inputs(1, 200, 200, 64, 1, 128, 777)
    o, lse = prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=0.09, out_dtype=out_dtype, packed=True)
    sync_check()
    ro, rl = oracle.sdpa(q, k, v, True, 0.09)
    check_o(o.float().cpu().numpy(), ro, out_dtype == torch.bfloat16)
    check_lse(lse.cpu().numpy(), rl)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(128, 1), (64, 2), (32, 1), (16, 2), (8, 1),
                                    (28, 4), (12, 1), (96, 1), (100, 2), (3, 3)])
def test_packed_decode(d, Hq, Hkv):
    """Head groups that divide 128 and groups that do not (7, 12, 96, 50, 1): the
    one-token decode's single position fills the first G rows of the tile."""
    # one KV tile (the second key half empty), two, odd counts (unequal halves),
    # ragged tails, an empty sequence
    lens = torch.tensor([0, 1, 29, 128, 129, 300, 640, 1000, 2500, 77], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(len(lens), Hq, Hkv, d, lens, 600 + d + Hq)
    scale = 1.0 / np.sqrt(d)
    o, lse = decode_packed(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), scale, out_dtype=torch.float32)
    sync_check()
    ro, rl = oracle.decode(q, kc, vc, lens, scale)
    check_o(o.cpu().numpy(), ro, False)
    check_lse(lse.cpu().numpy(), rl)


def test_packed_decode_cache_rows_past_length_ignored():
    lens = torch.tensor([100, 3], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(2, 16, 1, 128, lens, 611, Lmax=400)
    kc[:, 100:] = 40.0
    vc[:, 100:] = -40.0
    o, lse = decode_packed(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), 0.1, out_dtype=torch.float32)
    sync_check()
    ro, rl = oracle.decode(q, kc, vc, lens, 0.1)
    check_o(o.cpu().numpy(), ro, False)
    check_lse(lse.cpu().numpy(), rl)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(128, 1), (16, 2), (28, 4), (100, 1)])
@pytest.mark.parametrize("n_splits,min_rows", [(1, 1), (3, 1), (8, 256), (16, 64)])
def test_packed_decode_split_partials(d, Hq, Hkv, n_splits, min_rows):
    """Partials with the decode split rule (empty splits included) against the
    oracle's split partials, then merged against the oracle's decode."""
    from attention_forward_tcgen05_gb300 import decode_split_packed, merge
    lens = torch.tensor([0, 1, 29, 300, 1000, 2049, 5], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(len(lens), Hq, Hkv, d, lens, 700 + d + n_splits)
    scale = 1.0 / np.sqrt(d)
    po, pl = decode_split_packed(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), n_splits, min_rows, scale)
    o, lse = merge(po, pl, torch.float32)
    sync_check()
    ro, rl = oracle.decode_split(q, kc, vc, lens, scale, n_splits, min_rows)
    got_o, got_l = po.cpu().numpy(), pl.cpu().numpy()
    assert np.array_equal(np.isneginf(got_l), np.isneginf(rl))
    assert np.all(got_o[np.isneginf(rl)] == 0)
    check_o(got_o, ro, False)
    check_lse(got_l, rl)
    fo, fl = oracle.decode(q, kc, vc, lens, scale)
    check_o(o.cpu().numpy(), fo, False)
    check_lse(lse.cpu().numpy(), fl)


def test_packed_decode_split_halves_with_different_maxima():
    """A split's two key halves see score maxima far apart (the second half's keys
    scaled up), so the merge of the halves inside each split unit rescales one of
    them by a large factor before the split's partial is written; the partials and
    their merge against the oracle."""
    from attention_forward_tcgen05_gb300 import decode_split_packed, merge
    lens = torch.tensor([1000, 777, 2049], dtype=torch.int32)
    q, kc, vc = W.decode_inputs(len(lens), 64, 1, 128, lens, 731)
    ramp = torch.linspace(0.2, 3.0, kc.shape[1]).view(1, -1, 1, 1)
    kc = (kc.float() * ramp).to(torch.bfloat16)
    q = (q.float() * 2.0).to(torch.bfloat16)
    scale = 0.25
    po, pl = decode_split_packed(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), 3, 128, scale)
    o, lse = merge(po, pl, torch.float32)
    sync_check()
    ro, rl = oracle.decode_split(q, kc, vc, lens, scale, 3, 128)
    check_o(po.cpu().numpy(), ro, False)
    check_lse(pl.cpu().numpy(), rl)
    fo, fl = oracle.decode(q, kc, vc, lens, scale)
    check_o(o.cpu().numpy(), fo, False)
    check_lse(lse.cpu().numpy(), fl)


def test_packed_decode_no_keys_with_splits():
    from attention_forward_tcgen05_gb300 import decode_split_packed
    lens = torch.zeros(3, dtype=torch.int32)
    q, kc, vc = W.decode_inputs(3, 8, 1, 64, lens, 721, Lmax=0)
    po, pl = decode_split_packed(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), 4, 1, 0.125)
    sync_check()
    assert np.all(po.cpu().numpy() == 0) and np.all(np.isneginf(pl.cpu().numpy()))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_packed_decode_gqa_1641(out_dtype):
    """The 1641-key GQA decode (7 query heads per KV head, a group that does not
    divide 128) on the tensor cores, bf16 O through the TMA store of the first 7
    rows, against the oracle's decode."""
    s = W.GQA_DECODE
    q, kc, vc, lens = W.decode_inputs_for(s)
    o, lse = decode_packed(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), s.scale, out_dtype=out_dtype)
    sync_check()
    ro, rl = oracle.decode(q, kc, vc, lens, s.scale)
    check_o(o.float().cpu().numpy(), ro, out_dtype == torch.bfloat16)
    check_lse(lse.cpu().numpy(), rl)
