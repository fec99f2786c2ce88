"""Prefill FMHA (tcgen05) against the fp64 oracle, through the C ABI.

Small and medium shapes are compared element by element (every head dim,
both output types, the edge cases of the masks and tiles); a launch too large
for the full oracle is compared on sampled rows that the oracle computes one
by one.  The benchmark's full-size workloads are compared element by element
in test_full_parity.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_tcgen05_gb300 import prefill, sync_check
from attention_forward_tcgen05_gb300 import workloads as W
from tests.tolerances import check_lse, check_o

pytestmark = pytest.mark.gpu


def _run(q, k, v, causal, scale, out_dtype):
    o, lse = prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, out_dtype=out_dtype)
    sync_check()  # a bounded pipeline wait that ran out would surface here
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _full_compare(B, Hq, Hkv, Sq, Skv, d, causal, scale, seed, out_dtype=torch.float32, amp=1.0):
    q, k, v = W.prefill_inputs(B, Hq, Hkv, Sq, Skv, d, seed)
    if amp != 1.0:
        q = (q.float() * amp).to(torch.bfloat16)
        k = (k.float() * amp).to(torch.bfloat16)
    o, lse = _run(q, k, v, causal, scale, out_dtype)
    ro, rl = oracle.sdpa(q, k, v, causal, scale)
    check_o(o, ro, out_dtype == torch.bfloat16)
    check_lse(lse, rl)


def test_tiny_mha_causal_f32():
    s = W.TINY
    _full_compare(s.B, s.Hq, s.Hkv, s.Sq, s.Skv, s.d, s.causal, s.scale, s.seed, torch.float32)


SHAPES = [
    # B, Hq, Hkv, Sq, Skv, causal
    (1, 2, 1, 129, 129, True),    # GQA 2:1, ragged tail (129 = 128 + 1)
    (1, 2, 2, 1, 1, True),        # single row
    (1, 2, 2, 127, 127, True),
    (1, 3, 3, 257, 257, True),    # two query tiles + one row
    (2, 4, 2, 300, 300, False),
    (1, 2, 1, 100, 333, True),    # Sq < Skv, bottom-right causal
    (1, 2, 2, 300, 130, True),    # Sq > Skv: leading rows have no key
    (1, 1, 1, 64, 1000, False),   # 8 KV tiles: O rescales across tiles
    (1, 2, 2, 5, 0, True),        # no keys at all
    (1, 4, 1, 384, 384, True),    # GQA 4:1, three full query tiles
]


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["o_f32", "o_bf16"])
def test_small_shapes(shape, d, out_dtype):
    B, Hq, Hkv, Sq, Skv, causal = shape
    _full_compare(B, Hq, Hkv, Sq, Skv, d, causal, 1.0 / math.sqrt(d), 77 + d + Sq, out_dtype)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_large_scores_force_rescale(d):
    # |scores| of several tens: the running max jumps by more than 2^8 between tiles
    _full_compare(1, 2, 2, 200, 700, d, False, 0.35, 5, torch.float32, amp=3.0)
    _full_compare(1, 2, 2, 260, 260, d, True, 0.35, 6, torch.float32, amp=3.0)


@pytest.mark.parametrize("d", [64, 128])
def test_causal_scores_growing_every_tile(d):
    """Key rows scaled up along the sequence, so that every later KV tile raises a
    row's maximum by more than 2^8: a tile exponentiated against the stale reference
    overflows the rescale bound and is done again with the new maximum, on every
    tile (the causal launch runs on the persistent kernel)."""
    q, k, v = W.prefill_inputs(1, 2, 2, 600, 600, d, 31)
    ramp = torch.linspace(1.0, 6.0, 600).view(1, 600, 1, 1)
    q = (q.float() * 2.0).to(torch.bfloat16)
    k = (k.float().abs() * ramp).to(torch.bfloat16)
    q = q.float().abs().to(torch.bfloat16)
    o, lse = _run(q, k, v, True, 0.5, torch.float32)
    ro, rl = oracle.sdpa(q, k, v, True, 0.5)
    check_o(o, ro, False)
    check_lse(lse, rl)


def test_deterministic():
    q, k, v = W.prefill_inputs(1, 4, 2, 333, 333, 128, 9)
    a = prefill(q.cuda(), k.cuda(), v.cuda(), causal=True)
    b = prefill(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def _sample_rows(B, Hq, Sq, n_random, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 2, 127, 128, 129, 255, 256, Sq // 2, Sq - 129, Sq - 128, Sq - 2, Sq - 1]
    rows = set()
    for i in fixed:
        if 0 <= i < Sq:
            rows.add((int(rng.integers(B)), int(rng.integers(Hq)), i))
    while len(rows) < len(fixed) + n_random:
        rows.add((int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(Sq))))
    return sorted(rows)


def _full_size(shape: W.PrefillShape, out_dtype, n_random=40):
    q, k, v = W.prefill_inputs_for(shape)
    o, lse = prefill(q.cuda(), k.cuda(), v.cuda(), causal=shape.causal, scale=shape.scale,
                     out_dtype=out_dtype)
    sync_check()
    rows = _sample_rows(shape.B, shape.Hq, shape.Sq, n_random, shape.seed)
    ro, rl = oracle.sdpa_rows(q, k, v, shape.causal, shape.scale, rows)
    idx_b = torch.tensor([r[0] for r in rows])
    idx_h = torch.tensor([r[1] for r in rows])
    idx_i = torch.tensor([r[2] for r in rows])
    go = o.float().cpu()[idx_b, idx_i, idx_h].numpy()
    gl = lse.cpu()[idx_b, idx_h, idx_i].numpy()
    check_o(go, ro, out_dtype == torch.bfloat16, f"{shape.name} O")
    check_lse(gl, rl, f"{shape.name} LSE")
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_many_heads_long_kv_d256():
    # 148 query tiles of 128 rows against 64 KV tiles each, with KV rows 75 KB apart
    shape = W.PrefillShape("d256_h148_kv8192", 1, 148, 148, 128, 8192, 256, False,
                           1.0 / 16.0, "bf16", 77)
    _full_size(shape, torch.bfloat16, n_random=16)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Sq,Skv", [(4096, 4096), (4000, 1400), (4096, 100)], ids=["4096", "4000x1400", "4096x100"])
def test_noncausal_last_wave_as_key_halves(d, Sq, Skv):
    """A non-causal launch whose last wave is at most half full runs that wave's
    units as 128-row halves whose two query tiles take the two key halves (merged
    in the epilogue).  The shape is chosen from the SM count so that the launch
    has a few more units than SMs; rows of the last units (the last head's upper
    query blocks, on both sides of each 128-row split) and of the first wave are
    compared with the oracle."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    S = Sq
    H = n_sm // 16 + 1                     # 16 query blocks per head: 16*H units
    units = 16 * H
    assert -(-Sq // 256) == 16 and units > n_sm and 0 < units % n_sm <= n_sm // 2
    # Sq = 4000: the last query block's second 128-row half is partial;
    # Skv = 1400: 11 key tiles, halves of 6 and 5 ending in a partial tile;
    # Skv = 100: one key tile, so the second half holds no keys
    q, k, v = W.prefill_inputs(1, H, H, Sq, Skv, d, 90 + d if Skv == Sq else 90 + d + Skv)
    scale = 1.0 / math.sqrt(d)
    for out_dtype in (torch.float32, torch.bfloat16):
        o, lse = prefill(q.cuda(), k.cuda(), v.cuda(), causal=False, scale=scale, out_dtype=out_dtype)
        torch.cuda.synchronize()
        sync_check()
        last = H - 1
        first_tail_block = 16 - units % n_sm  # query blocks of the last head run as halves from here
        r0 = first_tail_block * 256
        picks = sorted({0, 1, 127, 128, r0 - 1, r0, r0 + 1, r0 + 127, r0 + 128, r0 + 129, r0 + 255,
                        r0 + 256, 3000, S - 129, S - 128, S - 2, S - 1} & set(range(S)))
        rows = [(0, last, i) for i in picks] + [(0, 0, 0), (0, 0, S - 1), (0, H // 2, 2100)]
        ro, rl = oracle.sdpa_rows(q, k, v, False, scale, rows)
        got_o = np.stack([o[0, i, h].float().cpu().numpy() for _, h, i in rows])
        got_l = np.array([lse[0, h, i].item() for _, h, i in rows])
        check_o(got_o, ro, out_dtype == torch.bfloat16, f"O {out_dtype}")
        check_lse(got_l, rl, f"LSE {out_dtype}")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["o_f32", "o_bf16"])
def test_d512_causal_gqa_whole_output(out_dtype):
    """Head dim 512, causal GQA over 12 query tiles and a ragged tail: every output
    element of both O halves (the second recomputes S) and LSE against the oracle."""
    q, k, v = W.prefill_inputs(1, 8, 2, 1500, 1500, 512, 5120)
    scale = 1.0 / math.sqrt(512)
    o, lse = _run(q, k, v, True, scale, out_dtype)
    ro, rl = oracle.sdpa(q, k, v, True, scale)
    check_o(o, ro, out_dtype == torch.bfloat16)
    check_lse(lse, rl)


def test_d512_deterministic_and_halves_consistent():
    """Two launches give the same bits; the two O halves come from separate passes
    over the keys, so each is compared with the oracle on its own columns."""
    q, k, v = W.prefill_inputs(2, 4, 4, 300, 700, 512, 5121)
    a = prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, out_dtype=torch.float32)
    b = prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, out_dtype=torch.float32)
    sync_check()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    ro, rl = oracle.sdpa(q, k, v, True, 1.0 / math.sqrt(512))
    got = a[0].cpu().numpy()
    check_o(got[..., :256], ro[..., :256], False, "O columns [0, 256)")
    check_o(got[..., 256:], ro[..., 256:], False, "O columns [256, 512)")
    check_lse(a[1].cpu().numpy(), rl)


PERSIST_SHAPES = [
    # B, Hq, Hkv, Sq, Skv: causal launches with more units (256-row query blocks x
    # heads x batch) than SMs, so each CTA of the persistent kernel walks several
    (2, 8, 2, 2900, 2900),    # ragged last block: its second tile partly past the end
    (3, 20, 4, 1000, 1300),   # Sq < Skv (bottom-right), a last block with one tile
    (1, 64, 8, 1100, 700),    # Sq > Skv: rows and whole tiles without any key
    (1, 40, 40, 2048, 2048),  # MHA, whole blocks
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", PERSIST_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["o_f32", "o_bf16"])
def test_causal_many_units_per_cta(shape, d, out_dtype):
    """Causal prefill whose units outnumber the SMs: every output element against
    the oracle, for both output types (bf16 O leaves through the staging tile the
    two query tiles take in turn, fp32 O through direct stores)."""
    B, Hq, Hkv, Sq, Skv = shape
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert -(-Sq // 256) * Hq * B > n_sm
    _full_compare(B, Hq, Hkv, Sq, Skv, d, True, 1.0 / math.sqrt(d), 400 + d + Sq, out_dtype)
