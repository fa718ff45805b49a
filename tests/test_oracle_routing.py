"""Pins of the oracle's routing (top-k, softmax), grouping (histogram,
permutation) and slot-pool LRU against brute force, library routines, closed
forms and an independently written list simulator."""
import collections
import math

import numpy as np
import pytest

import moe_synth as S
import oracle


def _brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return order[:k]


@pytest.mark.parametrize("T,E,k", [(50, 8, 2), (40, 32, 4), (20, 128, 8), (10, 8, 8), (10, 8, 1)])
def test_topk_matches_full_sort(T, E, k):
    rng = np.random.default_rng(T * 1000 + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = oracle.route(lg, k)
    for t in range(T):
        assert ids[t].tolist() == _brute_topk(lg[t], k)


def test_topk_ties_lower_id_wins():
    rng = np.random.default_rng(5)
    lg = np.round(rng.standard_normal((200, 16)) * 2).astype(np.float32)  # many exact ties
    lg[0] = 1.0
    lg[1, :] = 0.0
    lg[1, 3] = -0.0
    ids, _ = oracle.route(lg, 4)
    assert ids[0].tolist() == [0, 1, 2, 3]
    assert ids[1].tolist() == [0, 1, 2, 3]  # -0 == +0
    for t in range(200):
        assert ids[t].tolist() == _brute_topk(lg[t], 4)


def test_softmax_closed_forms():
    # k = 1: the single weight is exactly 1
    lg = np.random.default_rng(0).standard_normal((30, 8)).astype(np.float32)
    _, w = oracle.route(lg, 1)
    assert np.all(w == 1.0)
    # logits (ln 3, 0): weights 3/4 and 1/4 exactly
    lg = np.array([[np.float32(math.log(3.0)), 0.0, -5.0]], np.float32)
    _, w = oracle.route(lg, 2)
    e = math.exp(float(lg[0, 1]) - float(lg[0, 0]))
    assert abs(w[0, 0] - 0.75) <= 2 ** -24 and abs(w[0, 1] - 0.25) <= 2 ** -25
    assert w[0, 0] == np.float32(1 / (1 + e)) and w[0, 1] == np.float32(e / (1 + e))
    # equal selected logits: uniform weights
    lg = np.zeros((1, 8), np.float32)
    _, w = oracle.route(lg, 8)
    assert np.all(w == np.float32(0.125))


@pytest.mark.parametrize("wid", [0, 3, 4])
def test_softmax_sums_to_one_and_is_ordered(wid):
    wl = S.WORKLOADS[wid]
    lg = S.logits(wl, 0)[:2000]
    ids, w = oracle.route(lg, wl.top_k)
    s = w.astype(np.float64).sum(1)
    assert np.all(np.abs(s - 1) <= wl.top_k * 2.0 ** -23)
    assert np.all(np.diff(w, axis=1) <= 0)  # rank order = descending weight
    sel = np.take_along_axis(lg, ids, 1).astype(np.float64)
    ref = np.exp(sel - sel[:, :1])
    ref /= ref.sum(1, keepdims=True)
    assert np.max(np.abs(w - ref)) <= 2.0 ** -24


@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (300, 32, 4), (1000, 128, 8), (3, 8, 8), (0, 8, 2)])
def test_hist_perm_vs_stable_argsort(T, E, k):
    rng = np.random.default_rng(T + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[:, 1] -= 3  # an under-used expert, likely an empty group at small T
    ids, _ = oracle.route(lg, k) if T else (np.zeros((0, k), np.int32), None)
    counts, offsets, perm, inv = oracle.hist_perm(ids, E)
    flat = ids.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(inv[perm], np.arange(T * k))


def test_prefill_loads_each_unique_expert_once_gptoss_3k():
    """tinyserve README, How it works item 6: grouping tokens by expert loads
    each unique expert once -- 32 loads per layer at 3K context (32 experts)."""
    wl = S.WORKLOADS[3]
    ids, _ = oracle.route(S.logits(wl, 0), wl.top_k)
    counts, _, _, _ = oracle.hist_perm(ids, wl.experts)
    assert int((counts > 0).sum()) == 32
    assert int(counts.sum()) == 3072 * 4


class ListLRU:
    """Independent recency-list simulator (move-to-front list, no stamps)."""

    def __init__(self, S_, E):
        self.S, self.E = S_, E
        self.order = collections.OrderedDict()  # expert -> slot, oldest first
        self.free = list(range(S_))
        self.hits = self.misses = self.evictions = 0

    def step(self, counts):
        U = [e for e in range(self.E) if counts[e] > 0]
        if len(U) > self.S:
            raise OverflowError
        for e in U:
            if e in self.order:
                self.order.move_to_end(e)
                self.hits += 1
        loads = []
        for e in U:
            if e in self.order:
                continue
            if self.free:
                s = min(self.free)
                self.free.remove(s)
            else:
                victim = next(iter(self.order))
                s = self.order.pop(victim)
                self.evictions += 1
            self.order[e] = s
            self.misses += 1
            loads.append((e, s))
        return loads

    def slot_map(self):
        m = np.full(self.E, -1, np.int32)
        for e, s in self.order.items():
            m[e] = s
        return m


@pytest.mark.parametrize("S_,E,k,steps,bias", [(8, 32, 4, 300, 1.2), (3, 8, 2, 200, 0.0),
                                               (1, 4, 1, 50, 0.0), (16, 128, 8, 60, 0.8)])
def test_lru_matches_list_simulator(S_, E, k, steps, bias):
    rng = np.random.default_rng(S_ * 7 + E)
    rank = rng.permutation(E) + 1
    a, b = oracle.LRUPool(S_, E), ListLRU(S_, E)
    for _ in range(steps):
        lg = (rng.standard_normal((1, E)) - bias * np.log(rank)).astype(np.float32)
        ids, _ = oracle.route(lg, k)
        counts = np.bincount(ids.reshape(-1), minlength=E)
        assert a.step(counts) == b.step(counts)
        assert np.array_equal(a.slot_map(), b.slot_map())
    c = a.counters()
    assert (c["hits"], c["misses"], c["evictions"]) == (b.hits, b.misses, b.evictions)


def test_lru_hand_cases():
    # cyclic stream of S+1 experts with k = 1: every access misses under LRU
    S_, E = 3, 8
    p = oracle.LRUPool(S_, E)
    for i in range(40):
        c = np.zeros(E, np.int32)
        c[i % (S_ + 1)] = 1
        p.step(c)
    assert p.counters() == dict(hits=0, misses=40, evictions=40 - S_)
    # all-repeat stream: misses only on the cold start
    p = oracle.LRUPool(4, 8)
    c = np.array([1, 0, 2, 0, 1, 0, 0, 3], np.int32)
    for _ in range(10):
        p.step(c)
    assert p.counters() == dict(hits=36, misses=4, evictions=0)
    # capacity 1: alternate two experts; each access evicts the other
    p = oracle.LRUPool(1, 2)
    for i in range(6):
        loads = p.step(np.array([i % 2 == 0, i % 2 == 1], np.int32))
        assert loads == [(i % 2, 0)]
    assert p.counters() == dict(hits=0, misses=6, evictions=5)
    # lowest free slot first, then the least recent
    p = oracle.LRUPool(2, 5)
    assert p.step(np.array([0, 0, 0, 1, 0])) == [(3, 0)]
    assert p.step(np.array([1, 0, 0, 0, 0])) == [(0, 1)]
    assert p.step(np.array([0, 0, 0, 1, 0])) == []          # touch 3
    assert p.step(np.array([0, 0, 1, 0, 0])) == [(2, 1)]    # evicts 0 (older)
    # more unique experts than slots cannot be served
    with pytest.raises(OverflowError):
        p.step(np.array([1, 1, 1, 0, 0]))


def test_resident_pool_is_all_hits():
    wl = S.WORKLOADS[1]
    p = oracle.LRUPool(wl.slots, wl.experts, preload=True)
    for step in range(20):
        ids, _ = oracle.route(S.logits(wl, 0, step), wl.top_k)
        assert p.step(np.bincount(ids.reshape(-1), minlength=wl.experts)) == []
    assert np.array_equal(p.slot_map(), np.arange(wl.experts))
    assert p.counters()["misses"] == 0
