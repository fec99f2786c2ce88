"""The head-dimension-512 prefill kernel's mbarrier protocol, modelled on the CPU.

The d = 512 kernel runs on CTA pairs: a cluster of two CTAs takes 256 query
rows of one head, and rank 0's MMA warp issues every MMA for both (M = 256).
O is computed in two column halves one after the other (S is recomputed for
the second), so the T = 2 n_kv tiles form one sequence: tile jj belongs to
phase jj // n_kv and key tile jj % n_kv.  Each CTA's TMA producer fills a ring
of slots with its own share of every item, in the order K(0) K(1) { V(jj)
K(jj + 2) }; both CTAs' copies of an item complete on rank 0's full barrier,
which rank 0's producer arms for both.  The MMA warp consumes the items in that
order, issuing S(0) S(1) { P(jj).V(jj) S(jj + 2) } (two S buffers, S(jj) in
buffer jj % 2, each with its own S and P barrier).  MMA completions are
multicast to the S, O, final and empty barriers of both CTAs; P.V(jj) completes
on O barrier jj % 2.  Each CTA's softmax warpgroup waits for S(jj), may rescale
O in phase 0 (waiting for P(jj-1).V(jj-1)), publishes P(jj) -- rank 1's warps
with remote arrivals on rank 0's P barrier, eight arrivals in all -- and at the
end of each phase waits for that phase's last P.V on the final barrier (its
phase-th phase) before reading the O half.  Signals that cross the pair arrive
late, each by a random delay of its own.

A wait tests a phase parity, so it is sound only if its barrier has completed
exactly the phases before the awaited one or that phase too.  The model runs
the schedule against exact mbarrier semantics with random TMA, MMA, softmax and
cross-SM latencies, checks every wait for soundness, that every copy lands in
the phase it was armed for, that no O half is read or overwritten early and
that the pipeline drains, and must catch the unsound variants kept as negative
cases.
"""
import heapq
import itertools
import random

import pytest

from tests.test_prefill_protocol import Bar

# ring items as built: 32 KB slots; a K item holds four 64-column panels of the
# CTA's 64 keys (two items per tile), a V item both 128-column chunks' panels
# (one item per tile and phase)
SLOTS, K_ITEMS, V_ITEMS = 3, 2, 1


class PairBar(Bar):
    """An mbarrier whose transaction count may go below zero for a while: the
    peer CTA's bytes can land before the owner arms the barrier for them."""

    def complete_tx(self, n):
        self.tx -= n
        self._check()


def simulate(n_kv, slots, seed, k_items=K_ITEMS, v_items=V_ITEMS, p_count=8, arm_both=True,
             wait_own_empty=True, o_bars=2, s_per_buffer=True, fin_parity_by_phase=True):
    """One randomised run of the pair schedule; AssertionError on an unsound wait,
    an early overwrite of O or a deadlock.  p_count: arrivals the P barriers
    expect; arm_both=False arms the full barrier for rank 0's bytes only;
    wait_own_empty=False lets rank 1's producer refill a slot without waiting;
    o_bars=1 completes every P.V on one O barrier instead of alternating two;
    s_per_buffer=False keys the S and P barriers by nothing (one of each for both
    S buffers); fin_parity_by_phase=False waits for the final barrier's phase 0 at
    the end of both phases."""
    rng = random.Random(seed)
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = PairBar(name, count)
        return bars[name]

    T = 2 * n_kv
    now = [0]
    events = []
    seq = itertools.count()
    mma_free = [0]
    epilogue_done = [[False, False], [False, False]]  # [phase][rank]
    pv_completed = [0]  # P.V groups the tensor core has finished (not their barrier arrivals)

    def at(time, fn):
        heapq.heappush(events, (time, next(seq), fn))

    def mma(dur):
        mma_free[0] = max(now[0], mma_free[0]) + dur

    def cross():  # latency of a signal that crosses to the other SM of the pair
        return rng.randint(0, 2500)

    def commit_both(name):  # multicast: arrives on the barrier of each CTA
        for r in range(2):
            b = bar((name, r) if isinstance(name, str) else name + (r,))
            at(mma_free[0] + (cross() if r == 1 else 0), b.arrive)

    def wait(b, parity, use):
        assert b.done in (use, use + 1), f"{b.name}: waiting for phase {use} with {b.done} done"
        return ("wait", b, parity)

    def sbuf(jj):  # key of tile jj's S and P barriers, and the index of its awaited phase
        return (jj & 1, jj >> 1) if s_per_buffer else (0, jj)

    def items():
        seq_ = [("K", 0)] * k_items + [("K", 1)] * k_items
        for jj in range(T):
            seq_ += [("V", jj)] * v_items
            if jj + 2 < T:
                seq_ += [("K", jj + 2)] * k_items
        return seq_

    def land(b, use, delay):
        def fn():
            # bytes of item use land while the barrier still collects that item
            assert b.done == use, f"{b.name}: bytes of use {use} landed with {b.done} phases done"
            b.complete_tx(1)
        at(now[0] + delay, fn)

    def producer(r):
        q = bar("q")
        if r == 0:
            q.expect_tx(2)
        land(q, 0, rng.randint(50, 3000) + (cross() if r == 1 else 0))
        for g, _ in enumerate(items()):
            s, u = g % slots, g // slots
            if u > 0 and (wait_own_empty or r == 0):
                yield wait(bar(("empty", s, r)), (u & 1) ^ 1, u - 1)
            full = bar(("full", s))
            if r == 0:
                full.expect_tx(2 if arm_both else 1)
            land(full, u, rng.randint(50, 3000) + (cross() if r == 1 else 0))
            yield ("sleep", rng.randint(0, 30))

    def mma_warp():
        yield wait(bar("q"), 0, 0)
        g = [0]

        def take():
            s, u = g[0] % slots, g[0] // slots
            yield wait(bar(("full", s)), u & 1, u)
            return s

        def issue_s(jj):
            for _ in range(k_items):
                s = yield from take()
                for _ in range(8):
                    mma(rng.randint(20, 80))
                commit_both(("empty", s))
                g[0] += 1
            commit_both(("S", sbuf(jj)[0]))

        def issue_pv(jj):
            key, u = sbuf(jj)
            yield wait(bar(("P", key), p_count), u & 1, u)
            if jj == n_kv:  # first P.V of phase 1 overwrites the O half of phase 0
                assert all(epilogue_done[0]), "O half of phase 0 overwritten before both CTAs read it"
            for _ in range(v_items):
                s = yield from take()
                for _ in range(8):
                    mma(rng.randint(20, 80))
                commit_both(("empty", s))
                g[0] += 1
            commit_both(("O", jj % o_bars))
            at(mma_free[0], lambda: pv_completed.__setitem__(0, pv_completed[0] + 1))
            if jj % n_kv == n_kv - 1:
                commit_both("Fin")

        yield from issue_s(0)
        yield from issue_s(1)
        for jj in range(T):
            yield from issue_pv(jj)
            if jj + 2 < T:
                yield from issue_s(jj + 2)

    def softmax(r):
        for jj in range(T):
            ph, j = divmod(jj, n_kv)
            key, u = sbuf(jj)
            yield wait(bar(("S", key, r)), u & 1, u)
            yield ("sleep", rng.randint(20, 400))
            if ph == 0 and j > 0 and rng.random() < 0.3:
                uo = (jj - 1) // o_bars
                yield wait(bar(("O", (jj - 1) % o_bars, r)), uo & 1, uo)
                yield ("sleep", rng.randint(20, 200))
            p = bar(("P", key), p_count)
            for _ in range(4):
                if r == 0:
                    p.arrive()
                else:
                    at(now[0] + cross(), p.arrive)
            if j == n_kv - 1:
                fu = ph if fin_parity_by_phase else 0
                yield wait(bar(("Fin", r)), fu & 1, fu)
                # the final commit tracks every MMA issued before it; its arrival may
                # overtake the O barrier's, which the epilogue does not read
                assert pv_completed[0] >= (ph + 1) * n_kv, "O half read before its last P.V completed"
                yield ("sleep", rng.randint(1000, 8000))
                epilogue_done[ph][r] = True
            elif rng.random() < 0.2:
                yield ("sleep", rng.randint(100, 4000))

    procs = [producer(0), producer(1), softmax(0), softmax(1), mma_warp()]
    blocked = {}
    finished = set()
    advanced = [0]

    def step(i):
        while True:
            if i in blocked:
                _, b, parity = blocked[i]
                if not b.ready(parity):
                    return
                del blocked[i]
            advanced[0] += 1
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
    for _ in range(2000000):
        while True:
            before = advanced[0]
            for i in list(blocked):
                step(i)
            if advanced[0] == before:
                break
        if len(finished) == len(procs) and not events:
            break
        if not events:
            raise AssertionError(f"deadlock: blocked on {[blocked[i][1].name for i in blocked]}")
        now[0], _, fn = heapq.heappop(events)
        fn()
    assert len(finished) == len(procs), "pipeline did not drain"
    for b in bars.values():  # every phase that was armed completed
        assert b.pending == b.count and b.tx == 0, f"{b.name}: left mid-phase"


# (slots, K items per tile, V items per tile and phase): 32 KB slots as built,
# 16 KB slots (two K panels or one V panel per item), 8 KB slots (one K panel or
# 64 keys of a V panel), shallower rings
RINGS = [(SLOTS, K_ITEMS, V_ITEMS), (6, 4, 2), (12, 8, 4), (2, 2, 1), (1, 4, 2), (4, 4, 2), (5, 8, 4)]


@pytest.mark.parametrize("n_kv", [1, 2, 3, 8, 17])
@pytest.mark.parametrize("ring", RINGS, ids=lambda r: "x".join(map(str, r)))
def test_d512_protocol_is_sound(n_kv, ring):
    slots, k_items, v_items = ring
    for seed in range(40):
        simulate(n_kv, slots, seed, k_items, v_items)


def test_d512_one_s_barrier_for_both_buffers_is_unsound():
    """One S barrier and one P barrier for both S buffers: S(jj+1) can complete
    before the softmax waits for S(jj), two phases ahead.  The model must catch it."""
    failures = 0
    for seed in range(100):
        try:
            simulate(5, SLOTS, seed, s_per_buffer=False)
        except AssertionError:
            failures += 1
    assert failures > 0


def test_d512_final_barrier_waited_with_phase_zero_twice_is_unsound():
    """Waiting for the final barrier's phase 0 at the end of phase 1 too: the wait
    passes at once and the second O half would be read before its last P.V
    completed.  The model must catch it."""
    with pytest.raises(AssertionError):
        for seed in range(50):
            simulate(3, SLOTS, seed, fin_parity_by_phase=False)


def test_d512_p_barrier_counting_one_cta_is_unsound():
    """P barriers expecting four arrivals (one CTA's warps): P.V can start before
    the peer CTA has written its P.  The model must catch it."""
    with pytest.raises(AssertionError):
        for seed in range(50):
            simulate(3, SLOTS, seed, p_count=4)


def test_d512_full_barrier_armed_for_one_cta_is_unsound():
    """A full barrier armed for rank 0's bytes only completes without the peer's
    copy, whose bytes then land in a later phase.  The model must catch it."""
    with pytest.raises(AssertionError):
        for seed in range(50):
            simulate(3, SLOTS, seed, arm_both=False)


def test_d512_one_o_barrier_is_unsound_without_ordered_delivery():
    """Every P.V completing on one O barrier: the peer's copy of an O arrival can be
    overtaken by a later S arrival, and the softmax's rescale wait then tests a
    parity two phases ahead.  With two O barriers taken in turn the previous use of
    the awaited barrier lies a whole P.V and S group earlier.  The model must catch
    the one-barrier form."""
    with pytest.raises(AssertionError):
        for seed in range(200):
            for n_kv in (8, 17):
                simulate(n_kv, 6, seed, 4, 2, o_bars=1)


def test_d512_peer_refilling_without_its_empty_wait_is_unsound():
    """Rank 1's producer refilling a slot without waiting for its own empty
    barrier: its bytes land while the slot's previous item is still collected."""
    with pytest.raises(AssertionError):
        for seed in range(50):
            simulate(3, 2, seed, 2, 1, wait_own_empty=False)
