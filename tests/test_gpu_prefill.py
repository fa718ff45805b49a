"""GPU parity of the prefill expert path (moe_expert_ffn, MOE_PATH_PREFILL:
MXFP8 activations, tcgen05 block-scaled grouped GEMM) against the oracle:
rel-L2 <= 2e-3 and max-abs <= 1e-2 * rms(ref) on the layer output; MXFP8
codes and scales of the grouped activations bit-exact."""
import numpy as np
import pytest

import moe_synth as S
import oracle
from helpers import make_pool, rel_l2

pytestmark = pytest.mark.gpu

PREFILL_REL_L2 = 2e-3
PREFILL_MAX_ABS_RMS = 1e-2


def _check_prefill(out, ref):
    assert np.all(np.isfinite(out))
    rms = float(np.sqrt(np.mean(np.asarray(ref, np.float64) ** 2)))
    r = rel_l2(out, ref)
    m = float(np.max(np.abs(np.asarray(out, np.float64) - ref)))
    assert r <= PREFILL_REL_L2, r
    assert m <= PREFILL_MAX_ABS_RMS * rms, (m, rms)
    return r, m / rms


def _run_prefill(M, pool, wl, layer=0, step=0, tokens=None, logits=None):
    import torch

    lg = S.logits(wl, layer, step, tokens) if logits is None else logits
    T, E = lg.shape
    x = S.activations_bf16_bits(wl, layer, step, T)
    plan = M.RoutePlan.allocate(T, E, wl.top_k)
    M.moe_route_plan(torch.from_numpy(lg).cuda(), wl.top_k, plan, with_counts_host=False)
    slot_of = torch.from_numpy(pool.slot_map(layer).astype(np.int32)).cuda()
    ws = M.alloc_ffn_workspace(T, wl.top_k, wl.hidden, wl.inter, M.MOE_PATH_PREFILL)
    out = torch.empty((T, wl.hidden), dtype=torch.float32, device="cuda")
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    M.moe_expert_ffn(pool, layer, xt, plan, slot_of, out, ws, path=M.MOE_PATH_PREFILL)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lg, x, plan, ws


def _oracle_tokens(wl, lg, x, tokens, threads=16):
    ids, w = oracle.route(lg[tokens], wl.top_k)
    uniq = sorted(set(ids.reshape(-1).tolist()))
    ws = S.stack_experts(S.layer_weights(wl, 0, uniq))
    remap = {e: i for i, e in enumerate(uniq)}
    ids_r = np.vectorize(remap.get)(ids).astype(np.int32)
    return oracle.layer(x[tokens], ids_r, w, ws, prefill=True, threads=threads, want_intermediates=True)


def test_prefill_tiny():
    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[0]
    pool, host, dev = make_pool(M, wl)
    out, lg, x, plan, ws = _run_prefill(M, pool, wl)
    ref, it = _oracle_tokens(wl, lg, x, np.arange(wl.tokens))
    _check_prefill(out, ref)
    # grouped MXFP8 activations at the head of the workspace: bit-exact
    A, H = wl.tokens * wl.top_k, wl.hidden
    wsn = ws.cpu().numpy()
    xq = wsn[256:256 + A * H].reshape(A, H)
    perm = plan.perm.cpu().numpy()[:A]
    assert np.array_equal(xq, it["xq"][perm // wl.top_k])


@pytest.mark.parametrize("wid", [3, 4])
def test_prefill_full_size_sampled(wid):
    """GPT-OSS-shaped (3072 tokens, 32 experts, top-4) and Qwen-30B-A3B-shaped
    (16384 tokens, 128 experts, top-8, skewed groups) prefill at full size;
    the oracle recomputes 24 sampled tokens one by one."""
    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[wid]
    pool, host, dev = make_pool(M, wl)
    out, lg, x, plan, ws = _run_prefill(M, pool, wl)
    rng = np.random.default_rng(wid)
    tokens = np.sort(rng.choice(wl.tokens, 24, replace=False))
    tokens[0], tokens[-1] = 0, wl.tokens - 1
    ref, _ = _oracle_tokens(wl, lg, x, tokens)
    _check_prefill(out[tokens], ref)
    counts = plan.counts.cpu().numpy()
    if wid == 4:
        assert counts.max() > 4 * counts.min()  # uneven groups really are uneven


def test_prefill_edge_groups():
    """Empty expert groups, a group larger than one 128-row tile, a ragged
    last tile, assignments not a multiple of 32."""
    import routed_expert_ffn_histogram_gb300 as M

    wl = S.Workload(77, "edge_prefill", 1, 256, 512, 8, 3, 203, 1, 8, 0.0, 77)
    pool, host, dev = make_pool(M, wl)
    lg = S.logits(wl, 0)
    lg[:, 2] -= 20.0          # expert 2 never chosen
    lg[:150, 5] += 20.0       # expert 5 gets > 128 rows
    lg = lg.astype(np.float32)
    out, lg, x, plan, ws = _run_prefill(M, pool, wl, logits=lg)
    counts = plan.counts.cpu().numpy()
    assert counts[2] == 0 and counts[5] > 128
    ref, _ = _oracle_tokens(wl, lg, x, np.arange(wl.tokens))
    _check_prefill(out, ref)


def test_prefill_matches_decode_path_closely():
    """Both paths compute the same layer; they differ only by the MXFP8
    rounding of x and h (a few percent per element, ~1e-2 rel-L2)."""
    import routed_expert_ffn_histogram_gb300 as M
    from test_gpu_decode import _gpu_layer

    wl = S.WORKLOADS[0]
    pool, host, dev = make_pool(M, wl)
    out_p, lg, x, _, _ = _run_prefill(M, pool, wl)
    out_d = _gpu_layer(M, pool, 0, lg, x, wl.top_k, M.MOE_PATH_DECODE)
    assert rel_l2(out_p, out_d) < 0.1


@pytest.mark.parametrize("wid,slots,window,T", [(0, 4, 2, 16), (0, 6, 1, 16), (3, 8, 4, 64)])
def test_prefill_staged_small_pool(wid, slots, window, T):
    """Prefill through a pool with fewer slots than routed experts
    (moe_prefill_staged, windows staged on a copy stream): out within the
    prefill tolerance of the oracle and within fp32 atomic-order rounding of
    the resident-pool path; slot map and hit/miss/eviction counters
    bit-exact against the oracle's window events; every routed expert loaded
    at most once per call."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M
    from helpers import build_host_store

    wl = S.WORKLOADS[wid]
    E, k, H, I = wl.experts, wl.top_k, wl.hidden, wl.inter
    host, eb = build_host_store(M, wl, 1)
    dev = torch.empty(slots * eb, dtype=torch.uint8, device="cuda")
    pool = M.Pool(1, E, slots, H, I, host_experts=host, dev_slots=dev, policy="lru")
    lg = S.logits(wl, 0, 0, T)
    x = S.activations_bf16_bits(wl, 0, 0, T)
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    plan = M.RoutePlan.allocate(T, E, k, counts_host=True)
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_PREFILL)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    ref_pool = oracle.PolicyPool(slots, E, "lru")
    ref, _ = _oracle_tokens(wl, lg, x, np.arange(T))
    for call in range(2):
        with torch.cuda.stream(compute):
            M.moe_route_plan(torch.from_numpy(lg).cuda(), k, plan, stream=compute)
            pool.prefill_staged(0, plan.counts_host, window, k, x_bf16=xt, plan=plan, out=out, workspace=ws,
                                compute=compute, copy=copy)
        compute.synchronize()
        counts = plan.counts_host.numpy().copy()
        before = ref_pool.misses
        ref_pool.staged_prefill(counts, window)
        assert ref_pool.misses - before <= int((counts > 0).sum())
        _check_prefill(out.cpu().numpy(), ref)
        assert np.array_equal(pool.slot_map(0), ref_pool.slot_map())
        c, r = pool.counters(0), ref_pool.counters()
        assert (c["hits"], c["misses"], c["evictions"]) == (r["hits"], r["misses"], r["evictions"])
        assert c["h2d_bytes"] == c["misses"] * eb
    # the same routing on a fully resident pool
    dev_all = torch.empty(E * eb, dtype=torch.uint8, device="cuda")
    resident = M.Pool(1, E, E, H, I, host_experts=host, dev_slots=dev_all, preload=True)
    out2 = torch.empty_like(out)
    M.moe_expert_ffn(resident, 0, xt, plan, torch.arange(E, dtype=torch.int32, device="cuda"), out2, ws,
                     path=M.MOE_PATH_PREFILL)
    torch.cuda.synchronize()
    assert rel_l2(out.cpu().numpy(), out2.cpu().numpy()) <= 1e-6
    pool.close()
    resident.close()


@pytest.mark.parametrize("H,I", [(4096, 1024), (1024, 4096), (3584, 640)])
def test_prefill_reduction_lengths(H, I):
    """Prefill at the largest hidden and intermediate sizes the GEMM takes and
    at a reduction length whose last group of scale factors is partial
    (K = 640: five 128-K stages, one group of five; K = 3584: 28 stages,
    three groups of eight and one of four), against the oracle."""
    import routed_expert_ffn_histogram_gb300 as M

    wl = S.Workload(300 + H // 256 + I // 64, "prefill_k_sweep", 1, H, I, 8, 2, 260, 1, 8, 0.0,
                    300 + H // 256 + I // 64)
    pool, host, dev = make_pool(M, wl)
    out, lg, x, plan, ws = _run_prefill(M, pool, wl)
    ref, _ = _oracle_tokens(wl, lg, x, np.arange(wl.tokens))
    _check_prefill(out, ref)
