"""The decode kernel's shared-memory ring protocol, modelled on the CPU.

The decode kernel feeds its consumer warps through a ring of mbarrier-guarded
stages.  An mbarrier wait tests a phase *parity*, so a wait is only sound if
the waiter can never be two phases behind the barrier.  The kernel's rule:
every consumer warp reads every tile (the warps split the query heads, not
the rows), tile t lives in stage t % NS with use index t // NS, and a stage's
"empty" barrier counts one arrival per consumer warp -- so a stage is refilled
only after every consumer has released it, and each consumer waits on the
uses of a stage in order.  A second sound rule (each warp owning its own
stages) is checked too.

This test simulates producer, TMA completions (in random order) and consumers
against an exact model of mbarrier semantics (arrival count, transaction
bytes, phase parity) and checks that every wait wakes for the intended tile,
that no phase receives an extra arrival, and that the ring never deadlocks.
It also shows that the simpler rule "tile t -> stage t % n_stages" is unsound
whenever n_stages != NW (a consumer can wake on a stage's previous phase).
"""
import heapq
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "extra arrival on a phase"
        self._maybe_complete()

    def arrive_expect_tx(self, nbytes):
        self.tx += nbytes
        self.arrive()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        assert self.tx >= 0, "transaction count below zero"
        self._maybe_complete()

    def parity_done(self, parity):
        return (self.phase & 1) != parity


def owned_stage(t, NW, SPW):
    i = t // NW
    return (t % NW) * SPW + i % SPW, i // SPW


def round_robin_stage(t, NS):
    return t % NS, t // NS


def simulate(T, NW, stage_of, NS, seed, shared=False):
    """shared=False: warp w consumes tiles w, w+NW, ...; shared=True: every
    warp consumes every tile and a stage needs NW releases."""
    rng = random.Random(seed)
    full = [Bar(1) for _ in range(NS)]
    empty = [Bar(NW if shared else 1) for _ in range(NS)]
    content = [None] * NS
    releases = [0] * NS
    events, now, next_tile, done = [], 0, 0, 0
    cons = [{"i": 0, "t": None} for _ in range(NW)]
    step = 1 if shared else NW
    for _ in range(100000):
        moved = False
        if next_tile < T:
            s, k = stage_of(next_tile)
            if empty[s].parity_done((k & 1) ^ 1):
                full[s].arrive_expect_tx(1)
                heapq.heappush(events, (now + rng.randint(1, 30), 0, s, next_tile))
                next_tile += 1
                moved = True
        for w, c in enumerate(cons):
            t = c["i"] if shared else c["i"] * NW + w
            if c["t"] is None and t < T:
                s, k = stage_of(t)
                if full[s].parity_done(k & 1):
                    assert content[s] == t, f"warp {w} woke for tile {t}, stage {s} holds {content[s]}"
                    c["t"], c["s"] = t, s
                    heapq.heappush(events, (now + rng.randint(1, 30), 1, w, t))
                    moved = True
        if moved:
            continue
        if not events:
            break
        now, kind, a, t = heapq.heappop(events)
        if kind == 0:  # TMA landed in stage a
            content[a] = t
            full[a].complete_tx(1)
        else:  # warp a released its stage
            c = cons[a]
            releases[c["s"]] += 1
            if not shared or releases[c["s"]] == NW:
                content[c["s"]] = None
                releases[c["s"]] = 0
            empty[c["s"]].arrive()
            c["t"] = None
            c["i"] += 1
            done += 1
    assert done == (T * NW if shared else T), f"ring stalled after {done} tile releases"


@pytest.mark.parametrize("NW,SPW", [(4, 1), (4, 2), (3, 2), (2, 3)])
def test_owned_stages_are_sound(NW, SPW):
    for seed in range(150):
        for T in (1, 2, 5, 8, 17, 40):
            simulate(T, NW, lambda t: owned_stage(t, NW, SPW), NW * SPW, seed)


@pytest.mark.parametrize("NW,NS", [(1, 4), (2, 4), (4, 4), (4, 2), (4, 8), (3, 5)])
def test_shared_stages_are_sound(NW, NS):
    for seed in range(150):
        for T in (1, 2, 5, 8, 17, 40):
            simulate(T, NW, lambda t: round_robin_stage(t, NS), NS, seed, shared=True)


@pytest.mark.parametrize("NS", [3, 6])
def test_round_robin_stages_are_unsound(NS):
    failures = 0
    for seed in range(50):
        try:
            simulate(40, 4, lambda t: round_robin_stage(t, NS), NS, seed)
        except AssertionError:
            failures += 1
    assert failures > 0
