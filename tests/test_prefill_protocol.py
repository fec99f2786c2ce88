"""The prefill kernel's mbarrier protocol, modelled on the CPU.

The FMHA kernel coordinates a TMA producer warp, an MMA-issuing warp and one
softmax warpgroup per query tile through mbarriers whose waits test a phase
*parity*.  A wait is sound only if, when it starts, its barrier has completed
either exactly the phases before the awaited one or that phase too -- never
two phases more (the parity would then alias and the wait would never end).

This model restates each role's sequence of waits, arrivals and commits in
the kernel's order -- rings of K and V stages holding SUB KV tiles each
(waited for at their first tile, released after their last), two S buffers
per query tile with one S and one P barrier each (or one S buffer; or three
with S(j+2) issued ahead and two O barriers), the O and final barriers; per KV tile j the MMA warp issues S(j+1) for every query
tile, then P(j).V(j) for every query tile (with one S buffer: P_t(j).V(j)
then S_t(j+1), tile by tile) -- and runs it against exact mbarrier semantics with random TMA, MMA and
softmax latencies, including the optional O rescale.  It checks every wait
for soundness and that the pipeline always drains, for two query tiles (head
dims up to 128) and one (head dim 256), with causal (tile 0 shorter) and
ragged tile counts.
"""
import heapq
import itertools
import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.done = name, count, count, 0, 0

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: extra arrival"
        self._check()

    def expect_tx(self, n):
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        assert self.tx >= 0, f"{self.name}: tx below zero"
        self._check()

    def ready(self, parity):
        return (self.done & 1) != parity


def simulate(NQ, SK, SV, n_t, seed, p_per_buffer=True, NS=2, SUB=1, LOOK=1, NO=1, split=False):
    """Run one randomised schedule; raises AssertionError on an unsound wait or a deadlock.

    p_per_buffer=False keys the P barriers by query tile only (one barrier shared
    by both S buffers), the form whose parity can alias.  split=True gives the K
    ring and the V ring producers of their own, which fill their rings
    independently (the single-CTA kernel); otherwise one producer issues K stage
    jk before V stage jv while jk <= jv + LOOK (the CTA-pair kernel).
    """
    rng = random.Random(seed)
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(name, count)
        return bars[name]

    def p_bar(t, buf):
        return bar(("P", t, buf if p_per_buffer else 0), 4)

    def p_use(j):
        return j // NS if p_per_buffer else j

    # NO O barriers, P(j).V(j) completing on barrier j % NO (its (j // NO)-th phase)
    def o_bar(t, j):
        return bar(("O", t, j % NO))

    n = max(n_t)
    n_st = (n + SUB - 1) // SUB
    now = [0]
    events = []  # (time, seq, callback)
    seq = itertools.count()
    mma_free = [0]

    def at(time, fn):
        heapq.heappush(events, (time, next(seq), fn))

    def tma(b, nbytes):
        at(now[0] + rng.randint(50, 3000), lambda: b.complete_tx(nbytes))

    def mma(dur):
        mma_free[0] = max(now[0], mma_free[0]) + dur

    def commit(b):
        at(mma_free[0], b.arrive)

    def wait(b, parity, use):
        # use = index of the awaited phase; sound iff done in {use, use + 1}
        assert b.done in (use, use + 1), f"{b.name}: waiting for phase {use} with {b.done} done"
        return ("wait", b, parity)

    def producer_ring(kind, stages):
        for u in range(n_st):
            s, k = u % stages, u // stages
            if k > 0:
                yield wait(bar(("e" + kind, s)), (k & 1) ^ 1, k - 1)
            bar(("f" + kind, s)).expect_tx(1)
            tma(bar(("f" + kind, s)), 1)

    def producer_k():
        bar("q").expect_tx(1)
        tma(bar("q"), 1)
        yield from producer_ring("K", SK)

    def producer():
        bar("q").expect_tx(1)
        tma(bar("q"), 1)
        jk = jv = 0
        while jv < n_st:
            if jk < n_st and jk * SUB <= jv * SUB + LOOK:
                s, u = jk % SK, jk // SK
                if u > 0:
                    yield wait(bar(("eK", s)), (u & 1) ^ 1, u - 1)
                bar(("fK", s)).expect_tx(1)
                tma(bar(("fK", s)), 1)
                jk += 1
                continue
            s, u = jv % SV, jv // SV
            if u > 0:
                yield wait(bar(("eV", s)), (u & 1) ^ 1, u - 1)
            bar(("fV", s)).expect_tx(1)
            tma(bar(("fV", s)), 1)
            jv += 1

    def first(j):
        return j % SUB == 0

    def last(j):
        return j % SUB == SUB - 1 or j == n - 1

    def issue_s(t, j):
        for _ in range(8):
            mma(rng.randint(20, 80))
        commit(bar(("S", t, j % NS)))

    def issue_pv(t, j):
        use = p_use(j)
        yield wait(p_bar(t, j % NS), use & 1, use)
        for _ in range(4):
            mma(rng.randint(20, 80))
        commit(o_bar(t, j))
        if j == n_t[t] - 1:
            commit(bar(("Fin", t)))

    def mma_warp():
        yield wait(bar("q"), 0, 0)
        yield wait(bar(("fK", 0)), 0, 0)
        for t in range(NQ):
            if n_t[t] > 0:
                issue_s(t, 0)
        if last(0):
            commit(bar(("eK", 0)))
        # with LOOK > 1 (one query tile, NS = LOOK + 1 S buffers) the prologue also
        # issues S(1) .. S(LOOK - 1); the loop then issues S(j + LOOK) before P(j).V(j)
        for jj in range(1, LOOK):
            if jj < n:
                st = jj // SUB
                sn, un = st % SK, st // SK
                if first(jj):
                    yield wait(bar(("fK", sn)), un & 1, un)
                for t in range(NQ):
                    if jj < n_t[t]:
                        issue_s(t, jj)
                if last(jj):
                    commit(bar(("eK", sn)))
        for j in range(n):
            jn = j + LOOK
            if NS == 1:
                # one S buffer per tile: P_t(j).V(j), then S_t(j+1), tile by tile
                st = j // SUB
                s, u = st % SV, st // SV
                if first(j):
                    yield wait(bar(("fV", s)), u & 1, u)
                stn = jn // SUB
                sn, un = stn % SK, stn // SK
                k_ready = False
                for t in range(NQ):
                    if j < n_t[t]:
                        yield from issue_pv(t, j)
                    if jn < n_t[t]:
                        if not k_ready and first(jn):
                            yield wait(bar(("fK", sn)), un & 1, un)
                        k_ready = True
                        issue_s(t, jn)
                if k_ready and last(jn):
                    commit(bar(("eK", sn)))
                if last(j):
                    commit(bar(("eV", s)))
                continue
            if jn < n:
                st = jn // SUB
                sn, un = st % SK, st // SK
                if first(jn):
                    yield wait(bar(("fK", sn)), un & 1, un)
                for t in range(NQ):
                    if jn < n_t[t]:
                        issue_s(t, jn)
                if last(jn):
                    commit(bar(("eK", sn)))
            st = j // SUB
            s, u = st % SV, st // SV
            if first(j):
                yield wait(bar(("fV", s)), u & 1, u)
            for t in range(NQ):
                if j < n_t[t]:
                    yield from issue_pv(t, j)
            if last(j):
                commit(bar(("eV", s)))

    def softmax(t):
        for j in range(n_t[t]):
            buf, use = j % NS, j // NS
            yield wait(bar(("S", t, buf)), use & 1, use)
            yield ("sleep", rng.randint(20, 400))
            if j > 0 and rng.random() < 0.3:  # O rescale needs the previous P.V done
                u = (j - 1) // NO
                yield wait(o_bar(t, j - 1), u & 1, u)
                yield ("sleep", rng.randint(20, 200))
            for _ in range(4):  # one arrival per softmax warp
                p_bar(t, buf).arrive()
        if n_t[t] > 0:
            yield wait(bar(("Fin", t)), 0, 0)

    prods = [producer_k(), producer_ring("V", SV)] if split else [producer()]
    procs = prods + [softmax(t) for t in range(NQ)] + [mma_warp()]
    blocked = {}
    finished = set()
    advanced = [0]  # process steps taken

    def step(i):
        # advance process i until it blocks on a wait or sleeps
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
    for _ in range(200000):
        # step the blocked processes until none makes progress (an arrival made by
        # one of them can release another that was stepped before it)
        while True:
            before = advanced[0]
            for i in list(blocked):
                step(i)
            if advanced[0] == before:
                break
        if len(finished) == len(procs):
            break
        if not events:
            raise AssertionError(f"deadlock: blocked on {[blocked[i][1].name for i in blocked]}")
        now[0], _, fn = heapq.heappop(events)
        fn()
    assert len(finished) == len(procs), "pipeline did not drain"


CASES = [
    # query tiles, KV tiles per stage, K stages, V stages, KV tiles per query tile
    (2, 2, 2, 2, (9, 11)),   # d = 128, causal: tile 0 two KV tiles shorter
    (2, 2, 2, 2, (13, 13)),  # d = 128, non-causal, odd tile count
    (2, 2, 4, 4, (5, 6)),    # d = 64
    (2, 2, 2, 2, (0, 2)),    # first tile past the last query row
    (2, 2, 2, 2, (1, 1)),
    (2, 2, 2, 2, (1, 2)),
    (2, 2, 1, 1, (7, 8)),    # single-stage rings
    (1, 1, 3, 3, (11,)),     # CTA-pair kernel, d = 128: 3-stage rings
    (1, 1, 2, 2, (11,)),     # CTA-pair kernel, d = 256
    (1, 1, 1, 1, (9,)),      # d = 256
    (1, 1, 1, 1, (1,)),
    (1, 1, 1, 1, (2,)),
]
CASES_ONE_S = [
    # query tiles, KV tiles per stage, K stages, V stages, KV tiles per query tile
    (2, 1, 2, 2, (5, 6)),    # d = 128, causal: tile 0 one KV tile shorter
    (2, 1, 2, 2, (7, 7)),    # d = 128, non-causal
    (2, 1, 1, 1, (3, 4)),
    (2, 1, 2, 2, (0, 1)),
    (2, 1, 2, 2, (1, 1)),
    (2, 2, 2, 2, (5, 6)),
]


@pytest.mark.parametrize("NQ,SUB,SK,SV,n_t", CASES, ids=[str(c) for c in CASES])
def test_prefill_protocol_is_sound(NQ, SUB, SK, SV, n_t):
    for seed in range(120):
        simulate(NQ, SK, SV, list(n_t), seed, SUB=SUB)


CASES_LOOKAHEAD = [
    # CTA-pair kernel, d = 128: three S buffers, S(j+2) issued before P(j).V(j)
    # query tiles, K stages, V stages, KV tiles
    (1, 3, 3, (11,)),
    (1, 3, 3, (1,)),
    (1, 3, 3, (2,)),
    (1, 3, 3, (3,)),
    (1, 2, 2, (7,)),
    (1, 1, 1, (5,)),
]


@pytest.mark.parametrize("NQ,SK,SV,n_t", CASES_LOOKAHEAD, ids=[str(c) for c in CASES_LOOKAHEAD])
def test_prefill_protocol_three_s_buffers_is_sound(NQ, SK, SV, n_t):
    for seed in range(120):
        simulate(NQ, SK, SV, list(n_t), seed, NS=3, LOOK=2, NO=2)


def test_three_s_buffers_with_one_o_barrier_is_unsound():
    """With S(j+2) issued before P(j).V(j), the softmax of tile j can find
    P(j-2).V(j-2) still running; one O barrier would then be two phases behind
    the rescale's wait for P(j-1).V(j-1).  The model must catch this form."""
    failures = 0
    for seed in range(200):
        try:
            simulate(1, 3, 3, [11], seed, NS=3, LOOK=2, NO=1)
        except AssertionError:
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("NQ,SUB,SK,SV,n_t", CASES_ONE_S, ids=[str(c) for c in CASES_ONE_S])
def test_prefill_protocol_one_s_buffer_is_sound(NQ, SUB, SK, SV, n_t):
    for seed in range(120):
        simulate(NQ, SK, SV, list(n_t), seed, SUB=SUB, NS=1)


CASES_SPLIT = [
    # the single-CTA kernel: one S buffer per tile, K and V producers of their own
    # query tiles, K stages, V stages, KV tiles per query tile
    (2, 2, 3, (5, 6)),    # d = 128, causal
    (2, 2, 3, (13, 13)),  # d = 128, non-causal
    (2, 4, 4, (9, 10)),   # d = 64
    (2, 2, 3, (0, 1)),
    (2, 2, 3, (1, 1)),
    (2, 1, 1, (4, 5)),
    (2, 3, 1, (6, 6)),
]


@pytest.mark.parametrize("NQ,SK,SV,n_t", CASES_SPLIT, ids=[str(c) for c in CASES_SPLIT])
def test_prefill_protocol_split_producers_is_sound(NQ, SK, SV, n_t):
    for seed in range(120):
        simulate(NQ, SK, SV, list(n_t), seed, SUB=1, NS=1, split=True)


def simulate_slices(SK, SV, n, seed, NSL=2, NS=2):
    """CTA-pair schedule with independent key slices: NSL softmax warpgroups own
    slice h of every S tile with their own running max, sums and O accumulator;
    per KV tile j the MMA warp issues S(j+1), then P_h(j).V_h(j) for every slice
    (waiting for that slice's P barrier of S buffer j % NS), committing each to
    the slice's O barrier."""
    rng = random.Random(seed)
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(name, count)
        return bars[name]

    now = [0]
    events = []
    seq = itertools.count()
    mma_free = [0]

    def at(time, fn):
        heapq.heappush(events, (time, next(seq), fn))

    def tma(b):
        at(now[0] + rng.randint(50, 3000), lambda: b.complete_tx(1))

    def mma(dur):
        mma_free[0] = max(now[0], mma_free[0]) + dur

    def commit(b):
        at(mma_free[0], b.arrive)

    def wait(b, parity, use):
        assert b.done in (use, use + 1), f"{b.name}: waiting for phase {use} with {b.done} done"
        return ("wait", b, parity)

    def producer():
        bar("q").expect_tx(1)
        tma(bar("q"))
        jk = jv = 0
        while jv < n:
            if jk < n and jk <= jv + 1:
                s, u = jk % SK, jk // SK
                if u > 0:
                    yield wait(bar(("eK", s)), (u & 1) ^ 1, u - 1)
                bar(("fK", s)).expect_tx(1)
                tma(bar(("fK", s)))
                jk += 1
                continue
            s, u = jv % SV, jv // SV
            if u > 0:
                yield wait(bar(("eV", s)), (u & 1) ^ 1, u - 1)
            bar(("fV", s)).expect_tx(1)
            tma(bar(("fV", s)))
            jv += 1

    def issue_s(j):
        for _ in range(8):
            mma(rng.randint(20, 80))
        commit(bar(("S", j % NS)))

    def mma_warp():
        yield wait(bar("q"), 0, 0)
        yield wait(bar(("fK", 0)), 0, 0)
        issue_s(0)
        commit(bar(("eK", 0)))
        for j in range(n):
            if j + 1 < n:
                s, u = (j + 1) % SK, (j + 1) // SK
                yield wait(bar(("fK", s)), u & 1, u)
                issue_s(j + 1)
                commit(bar(("eK", s)))
            s, u = j % SV, j // SV
            yield wait(bar(("fV", s)), u & 1, u)
            for h in range(NSL):
                pu = j // NS
                yield wait(bar(("P", j % NS, h), 8), pu & 1, pu)
                for _ in range(4):
                    mma(rng.randint(20, 80))
                commit(bar(("O", h)))
            if j == n - 1:
                commit(bar("Fin"))
            commit(bar(("eV", s)))

    def softmax(h):
        for j in range(n):
            buf, use = j % NS, j // NS
            yield wait(bar(("S", buf)), use & 1, use)
            yield ("sleep", rng.randint(20, 600))
            if j > 0 and rng.random() < 0.3:  # this slice's O rescale needs P_h(j-1).V_h(j-1)
                yield wait(bar(("O", h)), (j - 1) & 1, j - 1)
                yield ("sleep", rng.randint(20, 200))
            for _ in range(8):  # 4 warps in each of the two CTAs
                bar(("P", buf, h), 8).arrive()
        if n > 0:
            yield wait(bar("Fin"), 0, 0)

    procs = [producer()] + [softmax(h) for h in range(NSL)] + [mma_warp()]
    blocked = {}
    finished = set()
    advanced = [0]  # process steps taken

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
    for _ in range(200000):
        # step the blocked processes until none makes progress (an arrival made by
        # one of them can release another that was stepped before it)
        while True:
            before = advanced[0]
            for i in list(blocked):
                step(i)
            if advanced[0] == before:
                break
        if len(finished) == len(procs):
            break
        if not events:
            raise AssertionError(f"deadlock: blocked on {[blocked[i][1].name for i in blocked]}")
        now[0], _, fn = heapq.heappop(events)
        fn()
    assert len(finished) == len(procs), "pipeline did not drain"


@pytest.mark.parametrize("SK,SV,n", [(3, 3, 11), (3, 3, 1), (3, 3, 2), (2, 2, 7), (1, 1, 5)])
def test_prefill_protocol_key_slices_is_sound(SK, SV, n):
    for seed in range(150):
        simulate_slices(SK, SV, n, seed)


def test_single_p_barrier_with_two_s_buffers_is_unsound():
    """One P barrier shared by both S buffers of a tile: the softmax can publish
    P(j+1) before the MMA warp has waited for P(j), two phases ahead of that
    wait.  The model must catch this form."""
    failures = 0
    for seed in range(200):
        try:
            simulate(1, 1, 1, [9], seed, p_per_buffer=False)
        except AssertionError:
            failures += 1
    assert failures > 0
