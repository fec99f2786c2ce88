"""The persistent prefill kernel's mbarrier protocol, modelled on the CPU.

One CTA walks a sequence of units; unit k has two query tiles with n0 and n1 KV
tiles (a causal unit has n1 = n0 + 1; a tile past the end or without keys has 0).
Roles and barriers, with their phases running on across units:
  * the Q warp: for each unit in which a tile has keys, waits until the tile's
    last S MMA of its previous such unit has completed (Qfree), then loads the
    tile's Q (Q barrier): both barriers count the tile's units with keys;
  * the K and V warps: one ring each, items in unit order, max(n0, n1) per unit;
  * the MMA warp: per unit waits for the Q tiles with keys and the first K item,
    issues S of both tiles, then per step V, and per tile P.V (after P) and the
    next S; it commits Qfree after a tile's last S of the unit, and Fin after its
    last P.V;
  * two softmax warpgroups: per unit and step wait S, maybe rescale (waiting for
    the previous P.V on O), publish P with four arrivals; then wait Fin (its phases
    count the tile's units with keys) and take the O staging tile in turn with the
    other tile (turn e = 2k + t waits for turn e - 1 to be read out).
The model checks every wait for soundness (its barrier has completed exactly the
phases before the awaited one, or that one too), that the pipeline drains, that
no S MMA of a unit is issued before its tile's Q has landed and that a tile's O
is not read before its last P.V completed, that no S MMA is issued over a P whose
P.V has not been issued, and that no unit's first P.V (which starts O afresh) is
issued before the tile's warpgroup has read out the previous unit's O.

A tcgen05.commit issued before the CTA's first MMA does not arrive (a CTA whose
first units had no keys timed out on its Q-free barrier): the model's commits
follow that rule.  The earlier form, Q and Q-free phases counted by unit with
key-less tiles completing them (a plain arrival on Q, a commit on Q-free), is
kept as a negative case: it needs that commit, and even with a plain arrival its
MMA warp can complete Q-free phases of consecutive key-less units two ahead of
the Q warp's wait.
"""
import heapq
import itertools
import random

import pytest

from tests.test_prefill_protocol import Bar


def simulate(units, SK, SV, seed, fin_by_unit=False, q_by_unit=None):
    """units: [(n0, n1), ...] of one CTA.  fin_by_unit=True waits for the final
    barrier with the unit index as its phase (wrong when a tile has no keys in
    some unit).  q_by_unit counts the Q and Q-free phases by unit, key-less tiles
    completing them with a commit ("commit") or a plain arrival ("arrive") on
    Q-free: the model must catch all three."""
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
    q_loaded = {}  # (t, k) -> True once that unit's Q tile landed

    def at(time, fn):
        heapq.heappush(events, (time, next(seq), fn))

    n_mma = [0]

    def mma(dur):
        mma_free[0] = max(now[0], mma_free[0]) + dur
        n_mma[0] += 1

    def commit(b):
        if n_mma[0] > 0:  # a commit before the first MMA never arrives
            at(mma_free[0], b.arrive)

    def wait(b, parity, use):
        assert b.done in (use, use + 1), f"{b.name}: waiting for phase {use} with {b.done} done"
        return ("wait", b, parity)

    def q_warp():
        m = [0, 0]
        for k, ns in enumerate(units):
            for t in range(2):
                if ns[t] == 0 and not q_by_unit:
                    continue
                ph = k if q_by_unit else m[t]
                if ph > 0:
                    yield wait(bar(("qfree", t)), (ph - 1) & 1, ph - 1)
                b = bar(("q", t))
                if ns[t] > 0:
                    b.expect_tx(1)

                    def land(b=b, t=t, k=k):
                        q_loaded[(t, k)] = True
                        b.complete_tx(1)
                    at(now[0] + rng.randint(100, 3000), land)
                    m[t] += 1
                else:
                    b.arrive()

    def ring_warp(kind, stages):
        g = 0
        for ns in units:
            for _ in range(max(ns)):
                s, u = g % stages, g // stages
                if u > 0:
                    yield wait(bar(("e" + kind, s)), (u & 1) ^ 1, u - 1)
                b = bar(("f" + kind, s))
                b.expect_tx(1)
                at(now[0] + rng.randint(50, 3000), lambda b=b: b.complete_tx(1))
                g += 1

    n_s = [0, 0]   # S MMAs issued per tile
    n_pv = [0, 0]  # P.V MMAs issued per tile
    o_read = [0, 0]  # units with keys whose O the tile's warpgroup has read out

    def mma_warp():
        gk = gv = 0
        J = [0, 0]
        m_pv = [0, 0]  # units with keys whose first P.V has been issued, per tile

        def issue_s(t, k):
            assert q_loaded.get((t, k)), f"S of tile {t} unit {k} issued before its Q landed"
            # S_t overwrites P_t of the tile's previous step: its P.V must be issued first
            assert n_pv[t] >= n_s[t], f"S of tile {t} issued over a P its P.V has not read"
            n_s[t] += 1
            for _ in range(8):
                mma(rng.randint(20, 80))
            commit(bar(("S", t)))

        mq = [0, 0]
        for k, ns in enumerate(units):
            n = max(ns)
            if n > 0:
                for t in range(2):
                    if ns[t] > 0:
                        ph = k if q_by_unit else mq[t]
                        yield wait(bar(("q", t)), ph & 1, ph)
                s, u = gk % SK, gk // SK
                yield wait(bar(("fK", s)), u & 1, u)
                for t in range(2):
                    if ns[t] > 0:
                        issue_s(t, k)
                        if ns[t] == 1:
                            commit(bar(("qfree", t)))
                commit(bar(("eK", s)))
                gk += 1
                for j in range(n):
                    sv, uv = gv % SV, gv // SV
                    yield wait(bar(("fV", sv)), uv & 1, uv)
                    k_ready = False
                    for t in range(2):
                        if j < ns[t]:
                            use = J[t] + j
                            yield wait(bar(("P", t), 4), use & 1, use)
                            if j == 0:  # this P.V starts O_t afresh: the last unit's O is out
                                assert o_read[t] >= m_pv[t], f"P.V into O of tile {t} before its O was read"
                                m_pv[t] += 1
                            n_pv[t] += 1
                            for _ in range(8):
                                mma(rng.randint(20, 80))
                            commit(bar(("O", t)))
                            if j == ns[t] - 1:
                                commit(bar(("Fin", t)))
                        if j + 1 < ns[t]:
                            if not k_ready:
                                s, u = gk % SK, gk // SK
                                yield wait(bar(("fK", s)), u & 1, u)
                                k_ready = True
                            issue_s(t, k)
                            if j + 2 == ns[t]:
                                commit(bar(("qfree", t)))
                    if k_ready:
                        commit(bar(("eK", gk % SK)))
                        gk += 1
                    commit(bar(("eV", sv)))
                    gv += 1
            for t in range(2):
                if ns[t] > 0:
                    mq[t] += 1
                elif q_by_unit == "commit":
                    commit(bar(("qfree", t)))
                elif q_by_unit == "arrive":
                    bar(("qfree", t)).arrive()
            J[0] += ns[0]
            J[1] += ns[1]

    o_done = [0, 0]  # P.V groups of each tile completed so far (from the O barrier)

    def softmax(t):
        J = F = 0
        for k, ns in enumerate(units):
            for j in range(ns[t]):
                use = J + j
                yield wait(bar(("S", t)), use & 1, use)
                yield ("sleep", rng.randint(20, 400))
                if j > 0 and rng.random() < 0.3:  # O rescale needs the previous P.V done
                    yield wait(bar(("O", t)), (use - 1) & 1, use - 1)
                    yield ("sleep", rng.randint(20, 200))
                for _ in range(4):
                    bar(("P", t), 4).arrive()
                if rng.random() < 0.15:
                    yield ("sleep", rng.randint(100, 3000))
            if ns[t] > 0:
                fu = k if fin_by_unit else F
                yield wait(bar(("Fin", t)), fu & 1, fu)
                # O is read now: every P.V of the tile up to this unit must have completed
                assert bar(("O", t)).done >= J + ns[t], f"O of tile {t} read before its last P.V completed"
                o_read[t] += 1
                F += 1
            e = 2 * k + t
            if e > 0:
                yield wait(bar("stg"), (e - 1) & 1, e - 1)
            yield ("sleep", rng.randint(200, 3000))  # rows into the staging tile, store, read out
            bar("stg").arrive()
            J += ns[t]

    procs = [q_warp(), ring_warp("K", SK), ring_warp("V", SV), mma_warp(), softmax(0), softmax(1)]
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
    for _ in range(1000000):
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


# unit sequences of one CTA: causal units (n, n + 1) of the heaviest-first order,
# non-causal ones (n, n), a last query block whose second tile lies past the end,
# units without keys, one-tile units
SEQUENCES = {
    "causal": [(25, 26), (11, 12), (1, 2)],
    "causal_long": [(25, 26), (23, 24), (5, 6), (3, 4), (1, 2)],
    "noncausal": [(16, 16), (16, 16), (16, 16)],
    "tail_past_end": [(13, 0), (4, 0), (7, 8)],
    "no_keys": [(0, 0), (3, 3), (0, 1), (2, 0), (0, 0)],
    "single": [(1, 1)],
    "ones": [(1, 2), (1, 1), (1, 0), (0, 1)],
    # units without keys before the CTA's first MMA (a packed schedule gives a CTA
    # only such units, or puts them first)
    "keyless_only": [(0, 0), (0, 0), (0, 0), (0, 0)],
    "keyless_first": [(0, 0), (0, 0), (2, 3), (0, 1)],
    "one_tile_first": [(0, 1), (1, 0), (0, 0)],
}
RINGS = [(2, 2), (4, 4), (1, 1), (3, 2)]


@pytest.mark.parametrize("name", list(SEQUENCES))
@pytest.mark.parametrize("SK,SV", RINGS, ids=[str(r) for r in RINGS])
def test_persistent_protocol_is_sound(name, SK, SV):
    for seed in range(40):
        simulate(SEQUENCES[name], SK, SV, seed)


def test_final_barrier_phase_by_unit_is_unsound():
    """Counting the final barrier's phases by unit instead of by the tile's units with
    keys goes wrong once a tile has no keys in some unit; the model must catch it."""
    with pytest.raises(AssertionError):
        for seed in range(40):
            simulate([(0, 2), (3, 3), (2, 2)], 2, 2, seed, fin_by_unit=True)


@pytest.mark.parametrize("units", [[(0, 0), (0, 0), (0, 0)], [(0, 0), (2, 3)]])
def test_commit_before_first_mma_is_caught(units):
    """Completing a key-less tile's Q-free phase with a commit before any MMA leaves
    the Q warp waiting forever on a CTA whose first units have no keys."""
    with pytest.raises(AssertionError):
        simulate(units, 2, 2, 0, q_by_unit="commit")


def test_key_less_units_racing_ahead_is_caught():
    """Counted by unit, consecutive key-less units let the MMA warp complete Q-free
    phases without waiting, two ahead of the Q warp's wait, whose parity then
    aliases."""
    with pytest.raises(AssertionError):
        for seed in range(40):
            simulate([(0, 0), (0, 0), (0, 0), (0, 0)], 2, 2, seed, q_by_unit="arrive")


def _unit_tiles(u, BH, Sq, Skv):
    """(n0, n1) of causal unit u: KV tiles of its two query tiles (0 past the end or
    without keys), as the kernel derives them."""
    nb = -(-Sq // 256)
    qb = nb - 1 - u // BH
    out = []
    for t in range(2):
        q0 = qb * 256 + t * 128
        if q0 >= Sq:
            out.append(0)
            continue
        hi = max(0, min(Skv, min(Sq, q0 + 128) - 1 + (Skv - Sq) + 1))
        out.append(-(-hi // 128))
    return tuple(out)


@pytest.mark.parametrize("BH,Sq,Skv", [(16, 2900, 2900), (60, 1000, 1300), (64, 1100, 700), (40, 2048, 2048),
                                       (28, 3314, 3314)])
def test_host_schedules_are_sound(BH, Sq, Skv):
    """The unit lists the host schedule gives 152 CTAs for the persistent-kernel test
    shapes and the 3314-row workload (CTAs with no units, with key-less units only,
    or key-less units first among them), each replayed through the model."""
    import attention_forward_tcgen05_gb300 as attn
    from attention_forward_tcgen05_gb300 import build as attn_build
    attn_build.build()
    attn.load()
    sched = attn.prefill_schedule(BH, Sq, Skv, True, 152)
    seqs = {tuple(_unit_tiles(u, BH, Sq, Skv) for u in lst) for lst in sched}
    for seq in seqs:
        for seed in range(8):
            simulate(list(seq), 4, 4, seed)
            simulate(list(seq), 2, 2, seed)
