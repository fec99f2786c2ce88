"""The key-halves decode schedule of the single-CTA kernel, modelled on the CPU.

With one query position per sequence both query tiles hold the same head rows
and take the two halves of the unit's n KV tiles: tile 0 the first
n0 = ceil(n / 2), tile 1 the rest.  The K and V rings run over items
i = (step i // 2, tile i % 2), each filled in item order by a TMA producer warp
of its own, independently of the other ring.  The MMA warp issues S of both
tiles' first items, then per step and tile P.V of the item and S of the tile's
next item.  Each softmax warpgroup waits for its S tiles, publishes P with four
arrivals, may rescale O (waiting for its previous P.V), waits for its last P.V
(Fin) -- and tile 1 then hands its row state to tile 0 through a named barrier,
after which tile 0 also waits for tile 1's Fin before reading O_1.

The model runs each role's waits, arrivals and commits against exact mbarrier
semantics with random TMA, MMA and softmax latencies and checks that every wait
is sound (its barrier at most one phase ahead) and that the pipeline drains.
"""
import heapq
import itertools
import random

import pytest

from tests.test_prefill_protocol import Bar


def simulate_halves(SK, SV, n, seed):
    rng = random.Random(seed)
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(name, count)
        return bars[name]

    n0 = (n + 1) // 2
    n_t = [n0, n - n0]
    now = [0]
    events = []
    seq = itertools.count()
    mma_free = [0]

    def at(time, fn):
        heapq.heappush(events, (time, next(seq), fn))

    def tma(b):
        at(now[0] + rng.randint(200, 6000), lambda: b.complete_tx(1))

    def mma(dur):
        mma_free[0] = max(now[0], mma_free[0]) + dur

    def commit(b):
        at(mma_free[0], b.arrive)

    def wait(b, parity, use):
        assert b.done in (use, use + 1), f"{b.name}: waiting for phase {use} with {b.done} done"
        return ("wait", b, parity)

    def producer_ring(kind, stages):
        # the K ring and the V ring have producers of their own and fill independently
        for u in range(n):
            s, k = u % stages, u // stages
            if k > 0:
                yield wait(bar(("e" + kind, s)), (k & 1) ^ 1, k - 1)
            bar(("f" + kind, s)).expect_tx(1)
            tma(bar(("f" + kind, s)))

    def producer():
        if n == 0:
            return
        bar("q").expect_tx(1)
        tma(bar("q"))
        yield from producer_ring("K", SK)

    def producer_v():
        if n == 0:
            return
        yield from producer_ring("V", SV)

    def issue_s(t):
        for _ in range(8):
            mma(rng.randint(20, 80))
        commit(bar(("S", t)))

    def mma_warp():
        if n == 0:
            return
        yield wait(bar("q"), 0, 0)
        ik = iv = 0
        for t in range(2):
            if n_t[t] > 0:
                s, u = ik % SK, ik // SK
                yield wait(bar(("fK", s)), u & 1, u)
                issue_s(t)
                commit(bar(("eK", s)))
                ik += 1
        for j in range(n0):
            for t in range(2):
                if j < n_t[t]:
                    s, u = iv % SV, iv // SV
                    yield wait(bar(("fV", s)), u & 1, u)
                    yield wait(bar(("P", t), 4), j & 1, j)
                    for _ in range(8):
                        mma(rng.randint(20, 80))
                    commit(bar(("O", t)))
                    if j == n_t[t] - 1:
                        commit(bar(("Fin", t)))
                    commit(bar(("eV", s)))
                    iv += 1
                if j + 1 < n_t[t]:
                    s, u = ik % SK, ik // SK
                    yield wait(bar(("fK", s)), u & 1, u)
                    issue_s(t)
                    commit(bar(("eK", s)))
                    ik += 1
        assert ik == n and iv == n

    def softmax(t):
        for j in range(n_t[t]):
            yield wait(bar(("S", t)), j & 1, j)
            yield ("sleep", rng.randint(200, 1600))
            if j > 0 and rng.random() < 0.3:  # O rescale: the previous P.V must be done
                yield wait(bar(("O", t)), (j - 1) & 1, j - 1)
                yield ("sleep", rng.randint(50, 300))
            for _ in range(4):
                bar(("P", t), 4).arrive()
        if n_t[t] > 0:
            yield wait(bar(("Fin", t)), 0, 0)
        if t == 1:
            bar("merge").arrive()  # always reached, whatever happened above
        else:
            yield wait(bar("merge"), 0, 0)
            if n_t[1] > 0:  # O_1 complete before tile 0 reads it
                yield wait(bar(("Fin", 1)), 0, 0)

    procs = [producer(), producer_v(), softmax(0), softmax(1), mma_warp()]
    blocked = {}
    finished = set()

    def step(i):
        while True:
            if i in blocked:
                _, b, parity = blocked[i]
                if not b.ready(parity):
                    return
                del blocked[i]
            try:
                req = next(procs[i])
            except StopIteration:
                finished.add(i)
                return
            if req[0] == "wait":
                blocked[i] = req
            elif req[0] == "sleep":
                at(now[0] + req[1], lambda i=i: step(i))
                return

    for i in range(len(procs)):
        step(i)
    for _ in range(400000):
        for i in list(blocked):
            step(i)
        if len(finished) == len(procs):
            break
        if not events:
            raise AssertionError(f"deadlock: blocked on {[blocked[i][1].name for i in blocked]}")
        now[0], _, fn = heapq.heappop(events)
        fn()
    assert len(finished) == len(procs), "pipeline did not drain"


# (K stages, V stages): d = 128 as built (3, 2), shallower rings (2, 2), (1, 1),
# d = 64 (5, 4)
RINGS = [(3, 2), (2, 2), (1, 1), (5, 4)]
# KV tiles of the unit: one (tile 1 empty), two, odd counts (unequal halves), long
TILES = [0, 1, 2, 3, 4, 5, 9, 16, 33]


@pytest.mark.parametrize("SK,SV", RINGS, ids=[str(r) for r in RINGS])
@pytest.mark.parametrize("n", TILES)
def test_halves_protocol_is_sound(SK, SV, n):
    for seed in range(60):
        simulate_halves(SK, SV, n, seed)
