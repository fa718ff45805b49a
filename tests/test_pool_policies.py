"""The library's slot pool (moe_pool_stage, dry-run mode: policy only, no
CUDA call) under each eviction policy, event by event against the oracle's
policy simulator: load lists, slot maps and hit/miss/eviction counters
bit-exact, on uniform and skewed routing streams, plus a checkpoint taken
mid-stream and restored into a fresh pool."""
import numpy as np
import pytest

import oracle
import routed_expert_ffn_histogram_gb300 as M


def _stream(rng, E, k, steps, bias):
    rank = rng.permutation(E) + 1
    for _ in range(steps):
        lg = rng.standard_normal(E) - bias * np.log(rank)
        top = np.argsort(-lg, kind="stable")[:k]
        c = np.zeros(E, np.int32)
        c[top] = 1
        yield c


@pytest.mark.parametrize("policy", oracle.POLICIES)
@pytest.mark.parametrize("S,E,k,bias", [(8, 32, 4, 1.2), (4, 16, 2, 0.0), (6, 64, 4, 0.8)])
def test_dry_run_pool_matches_oracle_policy(policy, S, E, k, bias):
    rng = np.random.default_rng(S * 1000 + E)
    layers = 2
    pool = M.Pool(layers, E, S, 256, 512, dry_run=True, policy=policy)
    ref = [oracle.PolicyPool(S, E, policy) for _ in range(layers)]
    for step, c in enumerate(_stream(rng, E, k, 400, bias)):
        layer = step % layers
        assert pool.stage(layer, c) == M.MOE_OK
        assert pool.last_loads(layer) == ref[layer].step(c)
        assert np.array_equal(pool.slot_map(layer), ref[layer].slot_map())
    for layer in range(layers):
        got, exp = pool.counters(layer), ref[layer].counters()
        assert (got["hits"], got["misses"], got["evictions"]) == (exp["hits"], exp["misses"], exp["evictions"])


@pytest.mark.parametrize("policy", oracle.POLICIES)
def test_policy_state_survives_checkpoint(policy):
    rng = np.random.default_rng(5)
    S, E, k = 4, 16, 2
    events = list(_stream(rng, E, k, 120, 0.5))
    a = M.Pool(1, E, S, 256, 512, dry_run=True, policy=policy)
    for c in events[:60]:
        a.stage(0, c)
    state = a.save()
    b = M.Pool(1, E, S, 256, 512, dry_run=True, policy=policy)
    assert b.load(state) == M.MOE_OK
    for c in events[60:]:
        a.stage(0, c)
        b.stage(0, c)
        assert a.last_loads(0) == b.last_loads(0)
    other = M.Pool(1, E, S, 256, 512, dry_run=True, policy=(M.MOE_POLICY_LRU if policy != "lru" else "fifo"))
    assert other.load(state) == M.MOE_ERR_STATE


def test_decode_only_staging_accounting():
    """A pool staging only the decode path's parts copies gate/up rows and
    the column-blocked down copy: fewer bytes per miss, same events."""
    E, S, H, I = 8, 4, 256, 512
    whole = M.Pool(1, E, S, H, I, dry_run=True)
    part = M.Pool(1, E, S, H, I, dry_run=True, stage_parts="decode")
    rng = np.random.default_rng(3)
    for c in _stream(rng, E, 2, 50, 0.0):
        whole.stage(0, c)
        part.stage(0, c)
        assert whole.last_loads(0) == part.last_loads(0)
    cw, cp = whole.counters(0), part.counters(0)
    eb = M.moe_expert_bytes(H, I)
    rs_gu = -(-(H // 2 + ((H // 32 + 15) // 16) * 16) // 32) * 32
    rs_d = -(-(I // 2 + ((I // 32 + 15) // 16) * 16) // 32) * 32
    d_off = 2 * I * rs_gu
    dt_off = -(-(d_off + H * rs_d) // 128) * 128
    assert cw["h2d_bytes"] == cw["misses"] * eb
    assert cp["h2d_bytes"] == cp["misses"] * (d_off + eb - dt_off)
    with pytest.raises(M.MoeError):
        M.Pool(1, E, S, H, I, dry_run=True, stage_parts=2)


def _prefill_counts(rng, E, k, T, bias):
    rank = rng.permutation(E) + 1
    c = np.zeros(E, np.int32)
    for _ in range(T):
        lg = rng.standard_normal(E) - bias * np.log(rank)
        c[np.argsort(-lg, kind="stable")[:k]] += 1
    return c


@pytest.mark.parametrize("policy", oracle.POLICIES)
@pytest.mark.parametrize("S,E,window", [(4, 16, 2), (6, 16, 3), (8, 32, 4), (8, 32, 1)])
def test_dry_run_staged_prefill_matches_oracle(policy, S, E, window):
    """moe_prefill_staged's staging (dry run) against the oracle's window
    events: slot maps after every call and counters bit-exact, one event per
    window, interleaved with ordinary decode-style events."""
    rng = np.random.default_rng(S * 100 + E + window)
    layers, k = 2, 2
    pool = M.Pool(layers, E, S, 256, 512, dry_run=True, policy=policy)
    ref = [oracle.PolicyPool(S, E, policy) for _ in range(layers)]
    windows = 0
    for call in range(40):
        layer = call % layers
        if call % 5 == 4:
            c = _prefill_counts(rng, E, k, 1, 1.0)    # a decode step in between
            assert pool.stage(layer, c) == M.MOE_OK
            ref[layer].step(c)
        else:
            T = int(rng.integers(1, 30))
            c = _prefill_counts(rng, E, k, T, 0.8)
            pool.prefill_staged(layer, c, window, k, T=T)
            windows += len(ref[layer].staged_prefill(c, window))
        assert np.array_equal(pool.slot_map(layer), ref[layer].slot_map())
    for layer in range(layers):
        got, exp = pool.counters(layer), ref[layer].counters()
        assert (got["hits"], got["misses"], got["evictions"]) == (exp["hits"], exp["misses"], exp["evictions"])
    assert pool.counters()["events"] == windows + 8


def test_staged_prefill_arguments():
    pool = M.Pool(1, 16, 6, 256, 512, dry_run=True)
    c = np.zeros(16, np.int32)
    c[[1, 5, 9]] = [2, 1, 1]
    with pytest.raises(M.MoeError) as e:
        pool.prefill_staged(0, c, 4, 2, T=2)          # window > S / 2
    assert e.value.status == M.MOE_ERR_INVALID
    with pytest.raises(M.MoeError) as e:
        pool.prefill_staged(0, c, 3, 2, T=3)          # counts do not sum to T * k
    assert e.value.status == M.MOE_ERR_INVALID
    pool.prefill_staged(0, c, 3, 2, T=2)
    assert pool.counters(0)["misses"] == 3
    dec = M.Pool(1, 16, 6, 256, 512, dry_run=True, stage_parts="decode")
    with pytest.raises(M.MoeError) as e:
        dec.prefill_staged(0, c, 3, 2, T=2)
    assert e.value.status == M.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("policy", oracle.POLICIES)
@pytest.mark.parametrize("S,E,k", [(4, 16, 2), (8, 32, 4)])
def test_dry_run_prefetch_matches_oracle(policy, S, E, k):
    """moe_pool_prefetch (dry run) between routing events of the next layer,
    against the oracle: slot maps and all counters bit-exact; a checkpoint
    taken mid-stream carries the routing frequencies and prefetch flags."""
    rng = np.random.default_rng(S + E)
    layers = 3
    pool = M.Pool(layers, E, S, 256, 512, dry_run=True, policy=policy)
    ref = [oracle.PolicyPool(S, E, policy) for _ in range(layers)]
    events = list(_stream(rng, E, k, 300, 1.0))
    for step, c in enumerate(events):
        layer = step % layers
        if step == 150:
            state = pool.save()
            pool = M.Pool(layers, E, S, 256, 512, dry_run=True, policy=policy)
            assert pool.load(state) == M.MOE_OK
        assert pool.stage(layer, c) == M.MOE_OK
        ref[layer].step(c)
        nxt, n = (layer + 1) % layers, int(rng.integers(0, 3))
        assert pool.prefetch(nxt, n) == len(ref[nxt].prefetch(n))
        assert np.array_equal(pool.slot_map(nxt), ref[nxt].slot_map())
    for layer in range(layers):
        got, exp = pool.counters(layer), ref[layer].counters()
        assert (got["hits"], got["misses"], got["evictions"]) == (exp["hits"], exp["misses"], exp["evictions"])
        pc = ref[layer].prefetch_counters()
        assert (got["prefetches"], got["prefetch_hits"]) == (pc["prefetches"], pc["prefetch_hits"])
    assert pool.counters()["prefetches"] > 0


def test_prefetch_arguments_and_no_op():
    pool = M.Pool(2, 8, 4, 256, 512, dry_run=True)
    with pytest.raises(M.MoeError) as e:
        pool.prefetch(2, 1)                       # layer out of range
    assert e.value.status == M.MOE_ERR_INVALID
    with pytest.raises(M.MoeError) as e:
        pool.prefetch(0, -1)
    assert e.value.status == M.MOE_ERR_INVALID
    assert pool.prefetch(0, 3) == 0               # nothing routed yet: no candidates
    c = np.zeros(8, np.int32)
    c[[1, 2]] = 1
    assert pool.stage(0, c) == M.MOE_OK
    before = pool.slot_map(0).copy()
    assert pool.prefetch(0, 0) == 0               # max_loads 0 changes nothing
    assert np.array_equal(pool.slot_map(0), before)
    assert pool.counters(0)["prefetches"] == 0


def test_staged_prefill_window_of_one_loads_each_expert_once():
    """Windows of one expert in a two-slot pool: every routed expert is its
    own event, none is loaded twice, and the last two stay resident."""
    pool = M.Pool(1, 8, 2, 256, 512, dry_run=True)
    ref = oracle.PolicyPool(2, 8, "lru")
    c = np.array([3, 0, 1, 2, 0, 0, 1, 1], np.int32)          # 5 routed experts, T*k = 8
    pool.prefill_staged(0, c, 1, 2, T=4)
    wins = ref.staged_prefill(c, 1)
    assert [w for w, _ in wins] == [[0], [2], [3], [6], [7]]
    got = pool.counters(0)
    assert got["misses"] == 5 and got["events"] == 5
    assert np.array_equal(pool.slot_map(0), ref.slot_map())
    assert sorted(int(e) for e in np.nonzero(pool.slot_map(0) >= 0)[0]) == [6, 7]
