"""Pins of the oracle's cache-policy simulator (oracle.PolicyPool) against
things other than itself: hand-worked event streams whose victim each
policy's reading fixes, chosen so that the policies disagree; the LRU mode
against the separately pinned C LRU step; and, on tiny streams, the fewest
misses any eviction choices could give (exhaustive search), which no policy
can beat.  Policies: tinyserve README, "Configuration" (cache_policy lru,
lfru, slru, lfu, fifo) and "How it works" item 3; events: Expert Offloading
topic page, replay-semantics study (one fused event per (layer, step))."""
import itertools

import numpy as np
import pytest

import oracle


def _ev(E, *experts):
    c = np.zeros(E, np.int32)
    for e in experts:
        c[e] += 1
    return c


def _run(policy, S, E, events):
    p = oracle.PolicyPool(S, E, policy)
    return p, [p.step(_ev(E, *ev)) for ev in events]


def test_fifo_ignores_rerouting_lru_does_not():
    # 0 loaded first, 1 second, 0 routed again, then 2 needs a slot
    events = [(0,), (1,), (0,), (2,)]
    _, fifo = _run("fifo", 2, 4, events)
    _, lru = _run("lru", 2, 4, events)
    assert fifo[-1] == [(2, 0)]      # evicts 0, the earliest load
    assert lru[-1] == [(2, 1)]       # evicts 1, routed longest ago


def test_lfu_and_lfru_prefer_frequency():
    # 0 routed twice, 1 once: both evict 1 even though 0 is older
    for pol in ("lfu", "lfru"):
        _, loads = _run(pol, 2, 4, [(0,), (0,), (1,), (2,)])
        assert loads[-1] == [(2, 1)], pol


def test_lfu_ties_by_id_lfru_ties_by_recency():
    # all routed once; load order 1, 0, 2 -> slots 0, 1, 2
    events = [(1,), (0,), (2,), (3,)]
    _, lfu = _run("lfu", 3, 5, events)
    _, lfru = _run("lfru", 3, 5, events)
    assert lfu[-1] == [(3, 1)]       # lowest id (0) sits in slot 1
    assert lfru[-1] == [(3, 0)]      # routed longest ago (1) sits in slot 0


def test_slru_protects_rerouted_experts():
    # S = 2: protected capacity 1.  0 is routed twice (protected), then the
    # scan 1, 2: SLRU evicts the probationary 1, LRU the older 0
    events = [(0,), (0,), (1,), (2,)]
    _, slru = _run("slru", 2, 4, events)
    _, lru = _run("lru", 2, 4, events)
    assert slru[-1] == [(2, 1)]
    assert lru[-1] == [(2, 0)]


def test_slru_demotes_the_least_recent_protected():
    # S = 4: capacity 2.  0, 1, 2, 3 loaded; 0, 1, 2 routed again in turn:
    # protecting 2 demotes 0 (routed longest ago), which counts as just
    # routed, so the next victim is 3
    p, _ = _run("slru", 4, 6, [(0,), (1,), (2,), (3,), (0,), (1,), (2,)])
    assert p.protected == {1, 2}
    assert p.step(_ev(6, 4)) == [(4, 3)]


def test_victims_are_never_routed_in_the_same_event():
    for pol in oracle.POLICIES:
        p, _ = _run(pol, 2, 4, [(0,), (1,)])
        loads = p.step(_ev(4, 0, 2))      # 0 is a hit; 2 must evict 1
        assert loads == [(2, 1)], pol
        with pytest.raises(OverflowError):
            p.step(_ev(4, 0, 1, 3))


def test_lru_mode_matches_the_c_lru_step():
    rng = np.random.default_rng(7)
    for S, E in [(2, 6), (4, 8), (8, 32)]:
        a, b = oracle.PolicyPool(S, E, "lru"), oracle.LRUPool(S, E)
        for _ in range(300):
            k = int(rng.integers(1, min(S, 4) + 1))
            ev = _ev(E, *rng.choice(E, size=k, replace=False))
            assert a.step(ev) == b.step(ev)
            assert np.array_equal(a.slot_map(), b.slot_map())
        assert a.counters() == b.counters()


def _fewest_misses(S, events):
    """Fewest misses over every choice of victims (exhaustive search)."""
    best = [10 ** 9]

    def go(i, resident, misses):
        if misses >= best[0]:
            return
        if i == len(events):
            best[0] = misses
            return
        U = set(events[i])
        need = sorted(U - resident)
        keep = resident & U
        others = sorted(resident - U)
        free = S - len(resident)
        n_evict = max(0, len(need) - free)
        for out in itertools.combinations(others, n_evict):
            go(i + 1, (resident - set(out)) | U, misses + len(need))

    go(0, frozenset(), 0)
    return best[0]


def test_no_policy_beats_the_offline_optimum_and_bookkeeping_holds():
    rng = np.random.default_rng(11)
    for _ in range(40):
        S, E = 2, 5
        events = [tuple(sorted(rng.choice(E, size=int(rng.integers(1, 3)), replace=False))) for _ in range(10)]
        opt = _fewest_misses(S, events)
        for pol in oracle.POLICIES:
            p, loads = _run(pol, S, E, events)
            c = p.counters()
            assert c["misses"] >= opt, (pol, events)
            assert c["hits"] + c["misses"] == sum(len(ev) for ev in events)
            assert c["misses"] >= len(set().union(*map(set, events)))
            assert sum(len(l) for l in loads) == c["misses"]


def test_staged_prefill_hand_worked_lru():
    """Six routed experts, four slots, windows of two, cold LRU pool: the
    first two windows fill the free slots; the third evicts the first
    window's experts (the oldest) and never the second window's."""
    p = oracle.PolicyPool(4, 6, "lru")
    got = p.staged_prefill(np.ones(6, np.int32), 2)
    assert [w for w, _ in got] == [[0, 1], [2, 3], [4, 5]]
    assert [loads for _, loads in got] == [[(0, 0), (1, 1)], [(2, 2), (3, 3)], [(4, 0), (5, 1)]]
    assert p.counters() == dict(hits=0, misses=6, evictions=2)


def test_staged_prefill_keeps_the_window_in_flight():
    """LFU would evict the just-loaded (once-used) experts of the previous
    window; the staged event must take the frequently used ones instead."""
    p = oracle.PolicyPool(4, 6, "lfu")
    for _ in range(3):
        p.step(_ev(6, 2, 3))          # 2 -> slot 0, 3 -> slot 1, three uses each
    got = p.staged_prefill(_ev(6, 0, 1, 4, 5), 2)
    assert got == [([0, 1], [(0, 2), (1, 3)]), ([4, 5], [(4, 0), (5, 1)])]
    # a plain event in the same state takes the once-used experts 0 and 1
    q = oracle.PolicyPool(4, 6, "lfu")
    for _ in range(3):
        q.step(_ev(6, 2, 3))
    q.step(_ev(6, 0, 1))
    assert q.step(_ev(6, 4, 5)) == [(4, 2), (5, 3)]


@pytest.mark.parametrize("policy", oracle.POLICIES)
def test_staged_prefill_invariants(policy):
    rng = np.random.default_rng(11)
    S, E = 6, 20
    p = oracle.PolicyPool(S, E, policy)
    for call in range(60):
        window = (1, 2, 3)[call % 3]
        counts = np.bincount(rng.choice(E, size=int(rng.integers(1, 40))), minlength=E).astype(np.int32)
        routed = [e for e in range(E) if counts[e] > 0]
        before = p.misses
        where = {e: int(s) for e, s in enumerate(p.slot_map()) if s >= 0}   # expert -> slot, replayed
        held = set()          # slots of the previous window's experts
        seen = []
        for win, loads in p.staged_prefill(counts, window):
            assert 1 <= len(win) <= window and all(counts[e] > 0 for e in win)
            assert all(e in win for e, _ in loads)
            for e, s in loads:
                assert s not in held                  # the window in flight keeps its slots
                where = {x: t for x, t in where.items() if t != s}
                where[e] = s
            assert all(e in where for e in win)       # the whole window is resident
            held = {where[e] for e in win}
            seen += win
        assert seen == routed                         # every routed expert in exactly one window
        assert p.misses - before <= len(routed)       # each routed expert loaded at most once
        assert where == {e: int(s) for e, s in enumerate(p.slot_map()) if s >= 0}


def test_prefetch_hand_worked_lru():
    """Two slots, LRU.  After routing 0, 1, 0, 2 the pool holds {0, 2};
    prefetching the next candidate (1, routed once) would have to evict 0
    (routed twice): declined.  After 1 is routed again it holds {1, 2};
    prefetch then loads 0 (routed twice) over 2 (once), and routing 0 next
    counts as a prefetch hit."""
    p = oracle.PolicyPool(2, 5, "lru")
    for ev in [(0,), (1,), (0,), (2,)]:
        p.step(_ev(5, *ev))
    assert p.slot_map().tolist() == [0, -1, 1, -1, -1]
    assert p.prefetch(1) == []
    p.step(_ev(5, 1))                     # evicts 0 (routed longest ago)
    assert p.slot_map().tolist() == [-1, 0, 1, -1, -1]
    assert p.prefetch(2) == [(0, 1)]      # over 2; experts 3, 4 never routed
    p.step(_ev(5, 0))
    assert p.prefetch_counters() == dict(prefetches=1, prefetch_hits=1)
    assert p.counters() == dict(hits=2, misses=4, evictions=3)


@pytest.mark.parametrize("policy", oracle.POLICIES)
def test_prefetch_invariants(policy):
    rng = np.random.default_rng(3)
    S, E = 4, 12
    p = oracle.PolicyPool(S, E, policy)
    for _ in range(300):
        c = np.zeros(E, np.int32)
        c[rng.choice(E, 2, replace=False, p=np.linspace(2, 1, E) / np.linspace(2, 1, E).sum())] = 1
        p.step(c)
        before = dict(p.slot_of)
        freq = list(p.freq)
        loads = p.prefetch(int(rng.integers(0, 3)))
        occupant = {s: e for e, s in before.items()}
        for e, s in loads:
            assert e not in before and freq[e] > 0
            v = occupant.get(s)
            assert v is None or freq[v] < freq[e]   # never displaces an expert routed as often or more
        assert p.prefetch_hits <= p.prefetches
