"""The causal prefill's unit schedule (host logic of the persistent launch; no GPU).

A unit is one 256-row query block of one (sequence, query head); unit u is query
block nb - 1 - u // BH of head u % BH.  Its cost is the KV steps of its longer
128-row query tile (one step per 128 keys it admits) plus a fixed per-unit
overhead.  The schedule must hand every unit to exactly one CTA, run each CTA's
units largest first, and leave no CTA more loaded than the wave deal it
replaces (units k*grid + c, every other wave reversed)."""
import math

import pytest

import attention_forward_tcgen05_gb300 as attn
from attention_forward_tcgen05_gb300 import build as attn_build

OVERHEAD = 3  # step-equivalents per unit the packing assumes


@pytest.fixture(scope="module", autouse=True)
def lib():
    attn_build.build()
    return attn.load()


def unit_steps(u, BH, Sq, Skv, causal):
    nb = math.ceil(Sq / 256)
    qb = nb - 1 - u // BH
    n = []
    for t in range(2):
        q0 = qb * 256 + t * 128
        if q0 >= Sq:
            n.append(0)
            continue
        if causal:
            last = min(Sq, q0 + 128) - 1 + (Skv - Sq)  # the tile's last row admits keys <= last
            kv_hi = max(0, min(Skv, last + 1))
        else:
            kv_hi = Skv
        n.append(math.ceil(kv_hi / 128))
    return max(n)


def wave_deal(units, grid):
    out = [[] for _ in range(grid)]
    for c in range(grid):
        k = 0
        while k * grid < units:
            u = k * grid + (grid - 1 - c if k & 1 else c)
            if u < units:
                out[c].append(u)
            k += 1
    return out


@pytest.mark.parametrize("BH,Sq,Skv,grid", [(28, 3314, 3314, 152), (28, 3314, 3314, 100), (1, 4096, 4096, 16),
                                           (64, 1000, 1000, 152), (8, 300, 2348, 152), (3, 8192, 8192, 152)])
def test_schedule_covers_every_unit_and_beats_the_wave_deal(BH, Sq, Skv, grid):
    sched = attn.prefill_schedule(BH, Sq, Skv, True, grid)
    units = math.ceil(Sq / 256) * BH
    assert sched is not None and len(sched) == grid
    assert sorted(u for lst in sched for u in lst) == list(range(units))
    cost = [unit_steps(u, BH, Sq, Skv, True) + OVERHEAD for u in range(units)]
    for lst in sched:  # largest first
        assert [cost[u] for u in lst] == sorted((cost[u] for u in lst), reverse=True)
    packed = max(sum(cost[u] for u in lst) for lst in sched)
    wave = max(sum(cost[u] for u in lst) for lst in wave_deal(units, grid))
    assert packed <= wave
    assert packed >= math.ceil(sum(cost) / grid)


def test_schedule_of_the_benchmark_workload():
    """3314 rows, 28 heads, 152 CTAs: the wave deal's most loaded CTA carries 47
    step-equivalents (3 per unit), the packing 42, against a mean of 40.7."""
    sched = attn.prefill_schedule(28, 3314, 3314, True, 152)
    cost = [unit_steps(u, 28, 3314, 3314, True) + OVERHEAD for u in range(364)]
    assert max(sum(cost[u] for u in lst) for lst in sched) == 42
    assert max(sum(cost[u] for u in lst) for lst in wave_deal(364, 152)) == 47


def test_schedule_is_deterministic():
    assert attn.prefill_schedule(28, 3314, 3314, True, 152) == attn.prefill_schedule(28, 3314, 3314, True, 152)


def test_many_units_per_cta_keep_the_wave_deal():
    # more than 64 units per CTA: nothing is written, the launch deals in waves
    assert attn.prefill_schedule(4 * 152, 65 * 256, 65 * 256, True, 152) is None


def test_schedule_validation():
    import ctypes
    offs = (ctypes.c_int * 153)()
    units = (ctypes.c_int * 364)()
    f = attn.attn_prefill_schedule
    assert f(0, 3314, 3314, 1, 152, offs, units, 364) == attn.ATTN_ERR_INVALID_ARG
    assert f(28, -1, 3314, 1, 152, offs, units, 364) == attn.ATTN_ERR_INVALID_ARG
    assert f(28, 3314, 3314, 1, 0, offs, units, 364) == attn.ATTN_ERR_INVALID_ARG
    assert f(28, 3314, 3314, 1, 152, None, units, 364) == attn.ATTN_ERR_INVALID_ARG
    assert f(28, 3314, 3314, 1, 152, offs, units, 363) == attn.ATTN_ERR_INVALID_ARG  # too small
    assert f(28, 3314, 3314, 1, 152, offs, units, 364) == 364
