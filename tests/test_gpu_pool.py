"""GPU parity of the offloaded decode (GPT-OSS shape, 8 of 32 slots per
layer, LRU, skewed routing): slot maps, load lists and hit/miss/eviction
counters bit-exact against the oracle's LRU for every (layer, step) event;
layer outputs computed from the staged slots match the oracle."""
import numpy as np
import pytest

import moe_synth as S
import oracle
from helpers import make_pool, rel_l2
from test_gpu_decode import DECODE_REL_L2, _oracle_layer

pytestmark = pytest.mark.gpu


def test_offload_decode_lru_and_outputs():
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[2]
    pool, host, dev = make_pool(M, wl, preload=False)
    ref = [oracle.LRUPool(wl.slots, wl.experts) for _ in range(wl.layers)]
    compute = torch.cuda.Stream()
    copy = torch.cuda.Stream()
    T, E, k, H, I = 1, wl.experts, wl.top_k, wl.hidden, wl.inter
    plan = M.RoutePlan.allocate(T, E, k, counts_host=True)
    slot_of = torch.empty(E, dtype=torch.int32, device="cuda")
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_DECODE)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    samples = {(0, 0), (3, 11), (7, 23)}
    with torch.cuda.stream(compute):
        for step in range(8):
            for layer in range(wl.layers):
                lg = torch.from_numpy(S.logits(wl, layer, step)).cuda()
                x = torch.from_numpy(S.activations_bf16_bits(wl, layer, step).view(np.int16)).cuda().view(
                    torch.bfloat16)
                M.moe_route_plan(lg, k, plan, stream=compute)
                assert pool.stage(layer, plan.counts_host, slot_of, compute=compute, copy=copy) == M.MOE_OK
                counts = plan.counts_host.numpy().copy()
                assert pool.last_loads(layer) == ref[layer].step(counts)
                assert np.array_equal(pool.slot_map(layer), ref[layer].slot_map())
                M.moe_expert_ffn(pool, layer, x, plan, slot_of, out, ws, path=M.MOE_PATH_DECODE, stream=compute)
                if (step, layer) in samples:
                    compute.synchronize()
                    got = out.cpu().numpy()
                    r, _ = _oracle_layer(wl, layer, step, prefill=False)
                    assert rel_l2(got, r) <= DECODE_REL_L2
    compute.synchronize()
    eb = M.moe_expert_bytes(H, I)
    for layer in range(wl.layers):
        c = pool.counters(layer)
        e = ref[layer].counters()
        assert (c["hits"], c["misses"], c["evictions"]) == (e["hits"], e["misses"], e["evictions"])
        assert c["h2d_bytes"] == e["misses"] * eb


def test_injected_copy_failure_on_device_pool():
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[0]
    pool, host, dev = make_pool(M, wl, slots=2, preload=False)
    counts = torch.zeros(8, dtype=torch.int32).pin_memory()
    slot_of = torch.full((8,), -7, dtype=torch.int32, device="cuda")
    counts[3] = 1
    pool.inject_copy_failures(1)
    with pytest.raises(M.MoeError):
        pool.stage(0, counts, slot_of)
    torch.cuda.synchronize()
    assert pool.slot_map(0).tolist() == [-1] * 8
    assert pool.counters(0)["errors"] == 1
    assert pool.stage(0, counts, slot_of) == M.MOE_OK
    torch.cuda.synchronize()
    assert slot_of.cpu().tolist() == [-1, -1, -1, 0, -1, -1, -1, -1]
    # slot 0 now holds expert 3's bytes
    eb = M.moe_expert_bytes(wl.hidden, wl.inter)
    assert torch.equal(dev[:eb].cpu(), host[3 * eb:4 * eb])


@pytest.mark.parametrize("policy", ["lfru", "slru"])
def test_offload_decode_only_staging(policy):
    """A pool that stages only what the fused decode kernel reads, under a
    non-LRU eviction policy: per (layer, step) event the load list and the
    slot map equal the oracle's policy simulation bit for bit, and so do the
    layer's hit/miss/eviction counters at the end; the layer outputs match
    the oracle; fewer bytes than whole experts are copied; the prefill path
    (which needs the skipped matrix) is refused."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[2]
    L = 3
    pool, host, dev = make_pool(M, wl, layers=L, preload=False)
    pool.close()
    pool = M.Pool(L, wl.experts, wl.slots, wl.hidden, wl.inter, host_experts=host, dev_slots=dev,
                  policy=policy, stage_parts="decode")
    ref = [oracle.PolicyPool(wl.slots, wl.experts, policy) for _ in range(L)]
    T, E, k, H, I = 1, wl.experts, wl.top_k, wl.hidden, wl.inter
    plan = M.RoutePlan.allocate(T, E, k, counts_host=True)
    slot_of = torch.empty(E, dtype=torch.int32, device="cuda")
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_DECODE)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(compute):
        for step in range(12):
            for layer in range(L):
                lg = torch.from_numpy(S.logits(wl, layer, step)).cuda()
                x = torch.from_numpy(S.activations_bf16_bits(wl, layer, step).view(np.int16)).cuda().view(
                    torch.bfloat16)
                M.moe_route_plan(lg, k, plan, stream=compute)
                assert pool.stage(layer, plan.counts_host, slot_of, compute=compute, copy=copy) == M.MOE_OK
                counts = plan.counts_host.numpy().copy()
                assert pool.last_loads(layer) == ref[layer].step(counts)
                assert np.array_equal(pool.slot_map(layer), ref[layer].slot_map())
                M.moe_expert_ffn(pool, layer, x, plan, slot_of, out, ws, path=M.MOE_PATH_DECODE, stream=compute)
                if step % 4 == 0 or step == 11:
                    compute.synchronize()
                    r, _ = _oracle_layer(wl, layer, step, prefill=False)
                    assert rel_l2(out.cpu().numpy(), r) <= DECODE_REL_L2
        compute.synchronize()
        for layer in range(L):
            c, e = pool.counters(layer), ref[layer].counters()
            assert (c["hits"], c["misses"], c["evictions"]) == (e["hits"], e["misses"], e["evictions"])
        c = pool.counters()
        assert c["evictions"] > 0
        assert 0 < c["h2d_bytes"] < c["misses"] * M.moe_expert_bytes(H, I)
        pws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_PREFILL)
        with pytest.raises(M.MoeError):
            M.moe_expert_ffn(pool, 0, x, plan, slot_of, out, pws, path=M.MOE_PATH_PREFILL, stream=compute)
    pool.close()


def test_offload_decode_with_prefetch():
    """Next-layer prefetch (moe_pool_prefetch) between each layer's staging
    and its FFN, on the copy stream: slot maps and all counters (including
    prefetches and prefetch hits) bit-exact against the oracle's policy
    simulation, and layer outputs that read prefetched experts match the
    oracle (the copies are ordered before their first reader)."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[2]
    L = 3
    pool, host, dev = make_pool(M, wl, layers=L, preload=False)
    pool.close()
    pool = M.Pool(L, wl.experts, wl.slots, wl.hidden, wl.inter, host_experts=host, dev_slots=dev, policy="lru")
    ref = [oracle.PolicyPool(wl.slots, wl.experts, "lru") for _ in range(L)]
    T, E, k, H, I = 1, wl.experts, wl.top_k, wl.hidden, wl.inter
    plan = M.RoutePlan.allocate(T, E, k, counts_host=True)
    slot_of = torch.empty(E, dtype=torch.int32, device="cuda")
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_DECODE)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    checked = 0
    with torch.cuda.stream(compute):
        for step in range(14):
            for layer in range(L):
                lg = torch.from_numpy(S.logits(wl, layer, step)).cuda()
                x = torch.from_numpy(S.activations_bf16_bits(wl, layer, step).view(np.int16)).cuda().view(
                    torch.bfloat16)
                M.moe_route_plan(lg, k, plan, stream=compute)
                assert pool.stage(layer, plan.counts_host, slot_of, compute=compute, copy=copy) == M.MOE_OK
                counts = plan.counts_host.numpy().copy()
                hits_before = ref[layer].prefetch_hits
                ref[layer].step(counts)
                nxt = (layer + 1) % L
                assert pool.prefetch(nxt, 2, compute=compute, copy=copy) == len(ref[nxt].prefetch(2))
                assert np.array_equal(pool.slot_map(nxt), ref[nxt].slot_map())
                M.moe_expert_ffn(pool, layer, x, plan, slot_of, out, ws, path=M.MOE_PATH_DECODE, stream=compute)
                if ref[layer].prefetch_hits > hits_before or step in (0, 13):
                    compute.synchronize()
                    r, _ = _oracle_layer(wl, layer, step, prefill=False)
                    assert rel_l2(out.cpu().numpy(), r) <= DECODE_REL_L2
                    checked += 1
    compute.synchronize()
    for layer in range(L):
        c, e, pc = pool.counters(layer), ref[layer].counters(), ref[layer].prefetch_counters()
        assert (c["hits"], c["misses"], c["evictions"]) == (e["hits"], e["misses"], e["evictions"])
        assert (c["prefetches"], c["prefetch_hits"]) == (pc["prefetches"], pc["prefetch_hits"])
    tot = pool.counters()
    assert tot["prefetch_hits"] > 0 and checked > 6
    pool.close()


@pytest.mark.parametrize("policy,parts,split", [("lru", "decode", False), ("fifo", "whole", False),
                                                ("lfu", "decode", False), ("lfru", "decode", False),
                                                ("slru", "decode", False), ("lru", "decode", True),
                                                ("slru", "whole", True)])
def test_offload_device_planned_staging(policy, parts, split):
    """Staging events planned on the GPU (moe_pool_stage_device) from the
    device counts, with the misses copied by the SMs out of the mapped host
    store: per (layer, step) event the slot map the planner writes equals
    the oracle's policy simulation; staged slots hold the host store's
    bytes; layer outputs match the oracle; after detaching, every layer's
    counters, last loads and slot map equal the oracle's.  Host staging
    before attaching and after detaching continues the same state.  With
    ``split`` the copies run on a second stream while the FFN of the event's
    hits runs (MOE_FFN_SKIP_ABSENT over the planner's hits map), and the
    loads' part is added after joining."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[2]
    L = 3
    pool, host, dev = make_pool(M, wl, layers=L, preload=False)
    pool.close()
    pool = M.Pool(L, wl.experts, wl.slots, wl.hidden, wl.inter, host_experts=host, dev_slots=dev,
                  policy=policy, stage_parts=parts)
    ref = [oracle.PolicyPool(wl.slots, wl.experts, policy) for _ in range(L)]
    T, E, k, H, I = 1, wl.experts, wl.top_k, wl.hidden, wl.inter
    eb = M.moe_expert_bytes(H, I)
    plan = M.RoutePlan.allocate(T, E, k, counts_host=True)
    slot_of = torch.empty(E, dtype=torch.int32, device="cuda")
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_DECODE)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    state = torch.zeros(pool.device_state_bytes(), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    copy_stream = torch.cuda.Stream()
    split_maps = torch.empty((2, E), dtype=torch.int32, device="cuda")
    last = [[] for _ in range(L)]
    with torch.cuda.stream(stream):
        for step in range(14):
            device_side = 4 <= step < 12
            if step == 4:
                pool.device_attach(state, stream=stream)
                with pytest.raises(M.MoeError):
                    pool.counters(0)
                counts_h = torch.zeros(E, dtype=torch.int32).pin_memory()
                with pytest.raises(M.MoeError):
                    pool.stage(0, counts_h, slot_of, compute=stream)
            if step == 12:
                assert pool.device_detach(stream=stream) == M.MOE_OK
                for layer in range(L):
                    c, e = pool.counters(layer), ref[layer].counters()
                    assert (c["hits"], c["misses"], c["evictions"]) == (e["hits"], e["misses"], e["evictions"])
                    assert pool.last_loads(layer) == last[layer]
                    assert np.array_equal(pool.slot_map(layer), ref[layer].slot_map())
            for layer in range(L):
                lg = torch.from_numpy(S.logits(wl, layer, step)).cuda()
                x = torch.from_numpy(S.activations_bf16_bits(wl, layer, step).view(np.int16)).cuda().view(
                    torch.bfloat16)
                M.moe_route_plan(lg, k, plan, stream=stream)
                if device_side:
                    if split:
                        pool.stage_device(layer, plan.counts, slot_of, split_dev=split_maps, stream=stream,
                                          copy=copy_stream)
                        M.moe_expert_ffn(pool, layer, x, plan, split_maps[0], out, ws, path=M.MOE_PATH_DECODE,
                                         stream=stream, skip_absent=True)
                        pool.device_join(layer, stream=stream)
                        M.moe_expert_ffn(pool, layer, x, plan, split_maps[1], out, ws, path=M.MOE_PATH_DECODE,
                                         stream=stream, skip_absent=True, accumulate=True)
                    else:
                        pool.stage_device(layer, plan.counts, slot_of, stream=stream)
                        M.moe_expert_ffn(pool, layer, x, plan, slot_of, out, ws, path=M.MOE_PATH_DECODE,
                                         stream=stream)
                    stream.synchronize()
                    counts = plan.counts_host.numpy().copy()
                    loads = ref[layer].step(counts)
                    last[layer] = loads
                    smap = ref[layer].slot_map()
                    assert np.array_equal(slot_of.cpu().numpy(), smap)
                    if split:
                        loaded = {e for e, _ in loads}
                        routed = counts > 0
                        want_hit = np.where(routed & ~np.isin(np.arange(E), list(loaded)), smap, -1)
                        want_load = np.where(np.isin(np.arange(E), list(loaded)), smap, -1)
                        got = split_maps.cpu().numpy()
                        assert np.array_equal(got[0], want_hit) and np.array_equal(got[1], want_load)
                    for e, s in loads:  # the staged parts, sampled at both ends of each
                        got = dev[(layer * wl.slots + s) * eb:(layer * wl.slots + s + 1) * eb]
                        want = host[((layer * E) + e) * eb:((layer * E) + e + 1) * eb]
                        assert torch.equal(got[:4096].cpu(), want[:4096])
                        assert torch.equal(got[-4096:].cpu(), want[-4096:])
                else:
                    assert pool.stage(layer, plan.counts_host, slot_of, compute=stream) == M.MOE_OK
                    counts = plan.counts_host.numpy().copy()
                    assert pool.last_loads(layer) == ref[layer].step(counts)
                    assert np.array_equal(pool.slot_map(layer), ref[layer].slot_map())
                    M.moe_expert_ffn(pool, layer, x, plan, slot_of, out, ws, path=M.MOE_PATH_DECODE,
                                     stream=stream)
                if step in (4, 7, 11, 13):
                    stream.synchronize()
                    r, _ = _oracle_layer(wl, layer, step, prefill=False)
                    assert rel_l2(out.cpu().numpy(), r) <= DECODE_REL_L2
        stream.synchronize()
    bpl = eb if parts == "whole" else None
    for layer in range(L):
        c, e = pool.counters(layer), ref[layer].counters()
        assert (c["hits"], c["misses"], c["evictions"]) == (e["hits"], e["misses"], e["evictions"])
        if bpl is not None:
            assert c["h2d_bytes"] == e["misses"] * bpl
    assert pool.counters()["evictions"] > 0
    pool.close()


def test_device_planned_capacity_and_negative_counts():
    """An event routing more experts than slots, or with a negative count,
    changes nothing on the device (no copies, the slot map stays) and is
    reported when the state is detached."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[0]
    pool, host, dev = make_pool(M, wl, slots=2, preload=False)
    E = wl.experts
    state = torch.zeros(pool.device_state_bytes(), dtype=torch.uint8, device="cuda")
    slot_of = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    pool.device_attach(state)
    counts[1] = 2
    pool.stage_device(0, counts, slot_of)
    torch.cuda.synchronize()
    assert slot_of.cpu().tolist() == [-1, 0] + [-1] * (E - 2)
    counts[2] = 1
    counts[5] = 3
    pool.stage_device(0, counts, slot_of)  # three routed, two slots
    torch.cuda.synchronize()
    assert slot_of.cpu().tolist() == [-1, 0] + [-1] * (E - 2)
    assert pool.device_detach() == M.MOE_ERR_CAPACITY
    assert pool.slot_map(0).tolist() == [-1, 0] + [-1] * (E - 2)
    c = pool.counters(0)
    assert (c["misses"], c["events"]) == (1, 1)
    assert pool.last_loads(0) == [(1, 0)]   # the last successful event's, as moe_pool_stage keeps them
    pool.device_attach(state)
    counts.zero_()
    counts[3] = -1
    pool.stage_device(0, counts, slot_of)
    assert pool.device_detach() == M.MOE_ERR_INVALID
    assert pool.counters(0)["events"] == 1
    pool.close()


def test_decode_ffn_skip_absent_parts_sum_to_the_layer():
    """MOE_FFN_SKIP_ABSENT: a layer's assignments served in two calls over
    complementary slot maps (the second accumulating) sum to the one-call
    result; a call that serves nothing leaves an accumulated out unchanged
    and writes zeros otherwise."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[1]
    pool, host, dev = make_pool(M, wl, layers=1, slots=wl.experts, preload=True)
    T, E, k, H, I = 1, wl.experts, wl.top_k, wl.hidden, wl.inter
    lg = torch.from_numpy(S.logits(wl, 0, 3)).cuda()
    x = torch.from_numpy(S.activations_bf16_bits(wl, 0, 3).view(np.int16)).cuda().view(torch.bfloat16)
    plan = M.RoutePlan.allocate(T, E, k)
    M.moe_route_plan(lg, k, plan, with_counts_host=False)
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_DECODE)
    full_map = torch.arange(E, dtype=torch.int32, device="cuda")
    full = torch.empty((T, H), dtype=torch.float32, device="cuda")
    M.moe_expert_ffn(pool, 0, x, plan, full_map, full, ws, path=M.MOE_PATH_DECODE)
    ids = plan.ids.cpu().numpy().ravel()
    a_map = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    b_map = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    for j, e in enumerate(ids):
        (a_map if j % 2 == 0 else b_map)[int(e)] = int(e)
    part = torch.empty((T, H), dtype=torch.float32, device="cuda")
    M.moe_expert_ffn(pool, 0, x, plan, a_map, part, ws, path=M.MOE_PATH_DECODE, skip_absent=True)
    M.moe_expert_ffn(pool, 0, x, plan, b_map, part, ws, path=M.MOE_PATH_DECODE, skip_absent=True,
                     accumulate=True)
    torch.cuda.synchronize()
    assert rel_l2(part.cpu().numpy(), full.cpu().numpy()) <= 1e-6
    r, _ = _oracle_layer(wl, 0, 3, prefill=False)
    assert rel_l2(part.cpu().numpy(), r) <= DECODE_REL_L2
    none = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    before = part.clone()
    M.moe_expert_ffn(pool, 0, x, plan, none, part, ws, path=M.MOE_PATH_DECODE, skip_absent=True, accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(part, before)
    M.moe_expert_ffn(pool, 0, x, plan, none, part, ws, path=M.MOE_PATH_DECODE, skip_absent=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(part).item() == 0
    pws = M.alloc_ffn_workspace(64, k, H, I, M.MOE_PATH_PREFILL)
    with pytest.raises(M.MoeError):
        M.moe_expert_ffn(pool, 0, x, plan, a_map, part, pws, path=M.MOE_PATH_PREFILL, skip_absent=True)
    pool.close()


def test_device_planned_step_in_cuda_graphs():
    """A decode step of device-planned staging (routing, planning, the copy
    on a second stream beside the hits' FFN, the loads' FFN) captured in a
    CUDA graph per step and replayed: counters, last loads and slot maps
    after detaching equal the oracle's LRU over the same events, and the
    replayed outputs match the oracle."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[2]
    L, steps = 3, 6
    pool, host, dev = make_pool(M, wl, layers=L, preload=False)
    pool.close()
    pool = M.Pool(L, wl.experts, wl.slots, wl.hidden, wl.inter, host_experts=host, dev_slots=dev, policy="lru",
                  stage_parts="decode")
    ref = [oracle.LRUPool(wl.slots, wl.experts) for _ in range(L)]
    T, E, k, H, I = 1, wl.experts, wl.top_k, wl.hidden, wl.inter
    lg = torch.stack([torch.stack([torch.from_numpy(S.logits(wl, l, g)) for l in range(L)])
                      for g in range(steps)]).cuda()
    xs = torch.stack([torch.stack([torch.from_numpy(S.activations_bf16_bits(wl, l, g).view(np.int16))
                                   for l in range(L)]) for g in range(steps)]).cuda().view(torch.bfloat16)
    outs = torch.zeros((steps, L, T, H), dtype=torch.float32, device="cuda")
    counts = torch.zeros((steps, L, E), dtype=torch.int32, device="cuda")
    plan = M.RoutePlan.allocate(T, E, k)
    slot_of = torch.empty(E, dtype=torch.int32, device="cuda")
    maps = torch.empty((2, E), dtype=torch.int32, device="cuda")
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_DECODE)
    state = torch.zeros(pool.device_state_bytes(), dtype=torch.uint8, device="cuda")
    stream, copy = torch.cuda.Stream(), torch.cuda.Stream()
    pool.device_attach(state, stream=stream)
    graphs = []
    for g in range(steps):
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=stream):
            for l in range(L):
                M.moe_route_plan(lg[g, l], k, plan, stream=stream, with_counts_host=False)
                counts[g, l].copy_(plan.counts)
                pool.stage_device(l, plan.counts, slot_of, split_dev=maps, stream=stream, copy=copy)
                M.moe_expert_ffn(pool, l, xs[g, l], plan, maps[0], outs[g, l], ws,
                                 path=M.MOE_PATH_DECODE, stream=stream, skip_absent=True)
                pool.device_join(l, stream=stream)
                M.moe_expert_ffn(pool, l, xs[g, l], plan, maps[1], outs[g, l], ws,
                                 path=M.MOE_PATH_DECODE, stream=stream, skip_absent=True, accumulate=True)
        graphs.append(cg)
    with torch.cuda.stream(stream):
        for cg in graphs:
            cg.replay()
    stream.synchronize()
    assert pool.device_detach(stream=stream) == M.MOE_OK
    c_host = counts.cpu().numpy()
    last = [[] for _ in range(L)]
    for g in range(steps):
        for l in range(L):
            last[l] = ref[l].step(c_host[g, l])
    for l in range(L):
        c, e = pool.counters(l), ref[l].counters()
        assert (c["hits"], c["misses"], c["evictions"]) == (e["hits"], e["misses"], e["evictions"])
        assert pool.last_loads(l) == last[l]
        assert np.array_equal(pool.slot_map(l), ref[l].slot_map())
    for g, l in ((0, 0), (steps - 1, L - 1), (3, 1)):
        r, _ = _oracle_layer(wl, l, g, prefill=False)
        assert rel_l2(outs[g, l].cpu().numpy(), r) <= DECODE_REL_L2
    assert pool.counters()["misses"] > 0
    pool.close()


def test_device_planned_events_after_host_prefetches():
    """Host steps (staging plus next-layer prefetch) alternate with
    device-planned steps: the experts a host prefetch copied in and an
    event then routes count as prefetch hits on the device too, and every
    counter (prefetches and prefetch hits included) and slot map equals the
    oracle's policy simulation of the same sequence."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[2]
    L = 3
    pool, host, dev = make_pool(M, wl, layers=L, preload=False)
    pool.close()
    pool = M.Pool(L, wl.experts, wl.slots, wl.hidden, wl.inter, host_experts=host, dev_slots=dev, policy="lru")
    ref = [oracle.PolicyPool(wl.slots, wl.experts, "lru") for _ in range(L)]
    T, E, k, H, I = 1, wl.experts, wl.top_k, wl.hidden, wl.inter
    plan = M.RoutePlan.allocate(T, E, k, counts_host=True)
    slot_of = torch.empty(E, dtype=torch.int32, device="cuda")
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_DECODE)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    state = torch.zeros(pool.device_state_bytes(), dtype=torch.uint8, device="cuda")
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    device_hits = 0
    with torch.cuda.stream(compute):
        for step in range(12):
            device_side = step % 2 == 1
            if device_side:
                before = pool.counters()["prefetch_hits"]
                pool.device_attach(state, stream=compute)
            for layer in range(L):
                lg = torch.from_numpy(S.logits(wl, layer, step)).cuda()
                x = torch.from_numpy(S.activations_bf16_bits(wl, layer, step).view(np.int16)).cuda().view(
                    torch.bfloat16)
                M.moe_route_plan(lg, k, plan, stream=compute)
                if device_side:
                    pool.stage_device(layer, plan.counts, slot_of, stream=compute)
                    compute.synchronize()
                    ref[layer].step(plan.counts_host.numpy().copy())
                    assert np.array_equal(slot_of.cpu().numpy(), ref[layer].slot_map())
                else:
                    assert pool.stage(layer, plan.counts_host, slot_of, compute=compute, copy=copy) == M.MOE_OK
                    ref[layer].step(plan.counts_host.numpy().copy())
                    nxt = (layer + 1) % L
                    assert pool.prefetch(nxt, 2, compute=compute, copy=copy) == len(ref[nxt].prefetch(2))
                M.moe_expert_ffn(pool, layer, x, plan, slot_of, out, ws, path=M.MOE_PATH_DECODE, stream=compute)
                if step in (1, 11) and layer == 1:
                    compute.synchronize()
                    r, _ = _oracle_layer(wl, layer, step, prefill=False)
                    assert rel_l2(out.cpu().numpy(), r) <= DECODE_REL_L2
            if device_side:
                assert pool.device_detach(stream=compute) == M.MOE_OK
                device_hits += pool.counters()["prefetch_hits"] - before
    compute.synchronize()
    for layer in range(L):
        c, e, pc = pool.counters(layer), ref[layer].counters(), ref[layer].prefetch_counters()
        assert (c["hits"], c["misses"], c["evictions"]) == (e["hits"], e["misses"], e["evictions"])
        assert (c["prefetches"], c["prefetch_hits"]) == (pc["prefetches"], pc["prefetch_hits"])
        assert np.array_equal(pool.slot_map(layer), ref[layer].slot_map())
    assert device_hits > 0
    pool.close()



@pytest.mark.parametrize("policy", ["lru", "fifo", "lfu", "lfru", "slru"])
def test_device_planned_random_events_match_host_planning(policy):
    """Random routing counts (including events that route more experts than
    slots) staged on the GPU and, for the same sequence, by a dry-run host
    pool: counters, slot maps and last loads of every layer agree after
    detaching, and the copied slots hold the host store's bytes."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[0]
    L, Sl, E = 2, 3, wl.experts
    pool, host, dev = make_pool(M, wl, layers=L, slots=Sl, preload=False)
    pool.close()
    pool = M.Pool(L, E, Sl, wl.hidden, wl.inter, host_experts=host, dev_slots=dev, policy=policy)
    ref = M.Pool(L, E, Sl, wl.hidden, wl.inter, dry_run=True, policy=policy)
    state = torch.zeros(pool.device_state_bytes(), dtype=torch.uint8, device="cuda")
    slot_of = torch.empty(E, dtype=torch.int32, device="cuda")
    counts_d = torch.empty(E, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(1234 + ["lru", "fifo", "lfu", "lfru", "slru"].index(policy))
    pool.device_attach(state)
    capacity_events = 0
    for i in range(80):
        layer = int(rng.integers(0, L))
        routed = rng.choice(E, size=int(rng.integers(0, Sl + 2)), replace=False)
        counts = np.zeros(E, np.int32)
        counts[routed] = rng.integers(1, 4, size=len(routed))
        counts_d.copy_(torch.from_numpy(counts))
        pool.stage_device(layer, counts_d, slot_of)
        rc = ref.stage(layer, torch.from_numpy(counts))
        capacity_events += rc == M.MOE_ERR_CAPACITY
    torch.cuda.synchronize()
    assert pool.device_detach() == (M.MOE_ERR_CAPACITY if capacity_events else M.MOE_OK)
    assert capacity_events > 0
    eb = M.moe_expert_bytes(wl.hidden, wl.inter)
    for layer in range(L):
        assert pool.counters(layer) == {**ref.counters(layer), "errors": pool.counters(layer)["errors"]}
        assert np.array_equal(pool.slot_map(layer), ref.slot_map(layer))
        assert pool.last_loads(layer) == ref.last_loads(layer)
        for e, s in enumerate(pool.slot_map(layer).tolist()):
            if s >= 0:
                got = dev[(layer * Sl + s) * eb:(layer * Sl + s + 1) * eb]
                want = host[(layer * E + e) * eb:(layer * E + e + 1) * eb]
                assert torch.equal(got.cpu(), want)
    pool.close()
    ref.close()


@pytest.mark.parametrize("policy,split", [("lru", True), ("slru", False)])
def test_route_stage_device_matches_route_then_stage(policy, split):
    """moe_pool_route_stage_device (routing and planning in one launch)
    against moe_route_plan followed by moe_pool_stage_device on a second
    pool over the same host store: per event the routing outputs (ids, w,
    counts, offsets, perm, inv), the slot map and the split maps are
    bit-exact; the staged slots and the layer outputs agree; after
    detaching, counters, last loads and slot maps are equal and equal to
    the oracle's policy simulation.  One step routes 8 tokens (32
    assignments, the most one launch takes), whose event overflows the 8
    slots in some layers: both pools then change nothing alike."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[2]
    L = 3
    pool_a, host, dev_a = make_pool(M, wl, layers=L, preload=False)
    pool_a.close()
    dev_b = torch.empty_like(dev_a)
    mk = lambda dev: M.Pool(L, wl.experts, wl.slots, wl.hidden, wl.inter, host_experts=host, dev_slots=dev,
                            policy=policy, stage_parts="decode")
    pool_a, pool_b = mk(dev_a), mk(dev_b)
    ref = [oracle.PolicyPool(wl.slots, wl.experts, policy) for _ in range(L)]
    E, k, H, I = wl.experts, wl.top_k, wl.hidden, wl.inter
    stream, copy_stream = torch.cuda.Stream(), torch.cuda.Stream()
    state_a = torch.zeros(pool_a.device_state_bytes(), dtype=torch.uint8, device="cuda")
    state_b = torch.zeros_like(state_a)
    with torch.cuda.stream(stream):
        pool_a.device_attach(state_a, stream=stream)
        pool_b.device_attach(state_b, stream=stream)
        for step in range(6):
            T = 8 if step == 3 else 1
            plan_a = M.RoutePlan.allocate(T, E, k, counts_host=True)
            plan_b = M.RoutePlan.allocate(T, E, k)
            ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_DECODE)
            slot_a = torch.empty(E, dtype=torch.int32, device="cuda")
            slot_b = torch.empty_like(slot_a)
            maps_a = torch.full((2, E), -7, dtype=torch.int32, device="cuda")
            maps_b = torch.full((2, E), -7, dtype=torch.int32, device="cuda")
            out_a = torch.empty((T, H), dtype=torch.float32, device="cuda")
            out_b = torch.empty_like(out_a)
            for layer in range(L):
                lg = torch.from_numpy(S.logits(wl, layer, step, tokens=T)).cuda()
                x = torch.from_numpy(S.activations_bf16_bits(wl, layer, step, tokens=T).view(np.int16)).cuda().view(
                    torch.bfloat16)
                M.moe_route_plan(lg, k, plan_a, stream=stream)
                cp = copy_stream if split else None
                pool_a.stage_device(layer, plan_a.counts, slot_a, split_dev=maps_a if split else None,
                                    stream=stream, copy=cp)
                pool_b.route_stage_device(layer, lg, k, plan_b, slot_b, split_dev=maps_b if split else None,
                                          stream=stream, copy=cp)
                stream.synchronize()
                copy_stream.synchronize()
                for f in ("ids", "w", "counts", "offsets", "perm", "inv"):
                    assert torch.equal(getattr(plan_a, f), getattr(plan_b, f)), f
                assert torch.equal(slot_a, slot_b)
                if split:
                    assert torch.equal(maps_a, maps_b)
                counts = plan_a.counts_host.numpy().copy()
                ok = counts.astype(bool).sum() <= wl.slots
                if ok:
                    ref[layer].step(counts)
                assert np.array_equal(slot_b.cpu().numpy(), ref[layer].slot_map())
                if T == 1:
                    for pool, dev, smap, out in ((pool_a, dev_a, slot_a, out_a), (pool_b, dev_b, slot_b, out_b)):
                        if split:
                            m = maps_a if pool is pool_a else maps_b
                            M.moe_expert_ffn(pool, layer, x, plan_a, m[0], out, ws, path=M.MOE_PATH_DECODE,
                                             stream=stream, skip_absent=True)
                            pool.device_join(layer, stream=stream)
                            M.moe_expert_ffn(pool, layer, x, plan_a, m[1], out, ws, path=M.MOE_PATH_DECODE,
                                             stream=stream, skip_absent=True, accumulate=True)
                        else:
                            M.moe_expert_ffn(pool, layer, x, plan_a, smap, out, ws, path=M.MOE_PATH_DECODE,
                                             stream=stream)
                        stream.synchronize()
                    r, _ = _oracle_layer(wl, layer, step, prefill=False)
                    assert rel_l2(out_a.cpu().numpy(), r) <= DECODE_REL_L2
                    assert rel_l2(out_b.cpu().numpy(), out_a.cpu().numpy()) <= 1e-6
        pool_a.device_join(L - 1, stream=stream)
        ra = pool_a.device_detach(stream=stream)
        rb = pool_b.device_detach(stream=stream)
    assert ra == rb
    eb = M.moe_expert_bytes(H, I)
    for layer in range(L):
        for s_ in pool_b.slot_map(layer):
            if s_ >= 0:  # the staged parts of each resident expert, sampled at both ends
                a0 = (layer * wl.slots + s_) * eb
                assert torch.equal(dev_a[a0:a0 + 4096], dev_b[a0:a0 + 4096])
                assert torch.equal(dev_a[a0 + eb - 4096:a0 + eb], dev_b[a0 + eb - 4096:a0 + eb])
    for layer in range(L):
        ca, cb, e = pool_a.counters(layer), pool_b.counters(layer), ref[layer].counters()
        assert ca == cb
        assert (ca["hits"], ca["misses"], ca["evictions"]) == (e["hits"], e["misses"], e["evictions"])
        assert pool_a.last_loads(layer) == pool_b.last_loads(layer)
        assert np.array_equal(pool_a.slot_map(layer), pool_b.slot_map(layer))
        assert np.array_equal(pool_b.slot_map(layer), ref[layer].slot_map())
    pool_a.close()
    pool_b.close()


def test_offload_loads_ffn_behind_the_copy():
    """The loaded experts' FFN on the copy stream right behind the copy
    kernel (launched programmatically after it), the hits' FFN beside the
    copy on the compute stream, both adding into a zeroed output with
    workspaces of their own, the compute stream joined to the copy stream
    by an event: layer outputs match the oracle and the counters and slot
    maps after detaching match the oracle's LRU."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[2]
    L = 3
    pool, host, dev = make_pool(M, wl, layers=L, preload=False)
    pool.close()
    pool = M.Pool(L, wl.experts, wl.slots, wl.hidden, wl.inter, host_experts=host, dev_slots=dev,
                  policy="lru", stage_parts="decode")
    ref = [oracle.PolicyPool(wl.slots, wl.experts, "lru") for _ in range(L)]
    E, k, H, I = wl.experts, wl.top_k, wl.hidden, wl.inter
    plan = M.RoutePlan.allocate(1, E, k, counts_host=True)
    slot_of = torch.empty(E, dtype=torch.int32, device="cuda")
    maps = torch.empty((2, E), dtype=torch.int32, device="cuda")
    ws_hits = M.alloc_ffn_workspace(1, k, H, I, M.MOE_PATH_DECODE)
    ws_loads = M.alloc_ffn_workspace(1, k, H, I, M.MOE_PATH_DECODE)
    out = torch.empty((1, H), dtype=torch.float32, device="cuda")
    state = torch.zeros(pool.device_state_bytes(), dtype=torch.uint8, device="cuda")
    stream, copy_stream = torch.cuda.Stream(), torch.cuda.Stream()
    joined = torch.cuda.Event()
    with torch.cuda.stream(stream):
        pool.device_attach(state, stream=stream)
        for step in range(8):
            for layer in range(L):
                lg = torch.from_numpy(S.logits(wl, layer, step)).cuda()
                x = torch.from_numpy(S.activations_bf16_bits(wl, layer, step).view(np.int16)).cuda().view(
                    torch.bfloat16)
                out.zero_()
                pool.route_stage_device(layer, lg, k, plan, slot_of, split_dev=maps, stream=stream,
                                        copy=copy_stream)
                M.moe_expert_ffn(pool, layer, x, plan, maps[0], out, ws_hits, path=M.MOE_PATH_DECODE,
                                 stream=stream, skip_absent=True, accumulate=True)
                M.moe_expert_ffn(pool, layer, x, plan, maps[1], out, ws_loads, path=M.MOE_PATH_DECODE,
                                 stream=copy_stream, skip_absent=True, accumulate=True)
                joined.record(copy_stream)
                stream.wait_event(joined)
                stream.synchronize()
                counts = np.bincount(plan.ids.cpu().numpy().ravel(), minlength=E).astype(np.int32)
                ref[layer].step(counts)
                assert np.array_equal(slot_of.cpu().numpy(), ref[layer].slot_map())
                if step in (0, 3, 7):
                    r, _ = _oracle_layer(wl, layer, step, prefill=False)
                    assert rel_l2(out.cpu().numpy(), r) <= DECODE_REL_L2
        assert pool.device_detach(stream=stream) == M.MOE_OK
    for layer in range(L):
        c, e = pool.counters(layer), ref[layer].counters()
        assert (c["hits"], c["misses"], c["evictions"]) == (e["hits"], e["misses"], e["evictions"])
        assert np.array_equal(pool.slot_map(layer), ref[layer].slot_map())
    assert pool.counters()["misses"] > 0
    pool.close()
