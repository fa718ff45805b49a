#!/usr/bin/env python
"""Benchmark of the routed-expert FFN layer on GB300.

Default workload: GPT-OSS-20B-shaped decode with every expert resident --
24 stacked MoE layers (hidden 2880, expert intermediate 2880, 32 experts,
top-4), one token per step, 768 distinct MXFP4 experts (10.2 GB) in the GPU
slot pool.  One step = one token through all 24 layers: routing (top-k,
softmax, histogram, permutation), the slot lookup, gate/up + SwiGLU, down,
and the weighted combine.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores on a bounded sample of the same workload instead.

Multi-GPU: the layer does not shard in this form (one token's four experts);
``--gpus N`` under torchrun runs N independent replicas and reports the sum.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import moe_synth as S  # noqa: E402

METRIC = "MoE-layer tokens/s; decode HBM GB/s & prefill TFLOPS as % of GB300 roofline"


# DRAM bytes per launch of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu capture of the kernel as it is built
# now; an entry goes back to None whenever that kernel changes.
NCU_TRAFFIC = {
    # one decode layer (2-layer decode capture; traffic per launch does not
    # depend on the number of layers)
    "decode_fused_kernel": 54_183_680 + 120_320,
    # gate/up launch + down launch of one 3072-token GPT-OSS-shaped layer
    "grouped_gemm_tc_kernel/gptoss20b_prefill_t3072": (320_057_856 + 30_262_784) + (232_777_984 + 29_761_536),
}

def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in [("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")]:
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


def replica_steps(rank: int, count: int, steps: int):
    """Decode steps (inputs) run by one replica: replicas are independent
    (the method is single-GPU; N GPUs run N decodes), so each rank takes
    its own sequence of the workload's steps."""
    return [(rank * 131 + g) % steps for g in range(count)]


def reduce_max_over_ranks(values, world: int, device="cpu"):
    """Largest of each value over all ranks (the job's time is the slowest
    rank's); identity on one process."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------------------
# oracle leg (CPU baseline / reference arm)
# --------------------------------------------------------------------------

def _oracle_token_sample(wl, step, layers, weights_cache, threads):
    """Time the oracle on `layers` of one decode step; returns seconds."""
    import oracle

    t0 = time.perf_counter()
    for l in layers:
        lg = S.logits(wl, l, step)
        ids, w = oracle.route(lg, wl.top_k)
        oracle.hist_perm(ids, wl.experts)
        x = S.activations_bf16_bits(wl, l, step)
        oracle.layer(x, ids, w, weights_cache[l], prefill=False, threads=threads)
    return time.perf_counter() - t0


def oracle_leg(wl, steps, layers_per_sample, threads):
    layers = list(range(0, wl.layers, max(1, wl.layers // layers_per_sample)))[:layers_per_sample]
    cache = {l: S.stack_experts(S.layer_weights(wl, l)) for l in layers}
    times = [_oracle_token_sample(wl, s, layers, cache, threads) for s in range(steps)]
    per_token = statistics.median(times) * wl.layers / len(layers)
    return 1.0 / per_token, layers, times


# --------------------------------------------------------------------------
# GPU leg
# --------------------------------------------------------------------------

def gpu_leg(args, wl, rank, world):
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    dev = torch.device("cuda", torch.cuda.current_device())
    L, E, k, H, I = wl.layers, wl.experts, wl.top_k, wl.hidden, wl.inter
    eb = M.moe_expert_bytes(H, I)

    # pinned host store of all experts (packed once), pool preloaded: resident
    host = torch.empty(L * E * eb, dtype=torch.uint8).pin_memory()
    for l in range(L):
        for e, w in enumerate(S.layer_weights(wl, l)):
            M.moe_pack_expert(w, H, I, host.data_ptr() + (l * E + e) * eb)
    slots = torch.empty(L * E * eb, dtype=torch.uint8, device=dev)
    pool = M.Pool(L, E, E, H, I, host_experts=host, dev_slots=slots, preload=True)
    slot_of = torch.arange(E, dtype=torch.int32, device=dev)

    G = args.warmup + args.steps
    step_ids = replica_steps(rank, G, wl.steps)
    lg_h = torch.from_numpy(np.stack([np.stack([S.logits(wl, l, s) for l in range(L)]) for s in step_ids]))
    x_h = torch.from_numpy(np.stack([np.stack([S.activations_bf16_bits(wl, l, s) for l in range(L)])
                                     for s in step_ids]).view(np.int16)).view(torch.bfloat16)
    lg_d = lg_h.to(dev)
    x_d = x_h.to(dev)
    residual = args.output == "residual"
    # overwrite: one output per (step, layer); residual: every layer of a
    # step adds into that step's residual-stream row (moe_decode_layer_acc)
    out_d = torch.zeros((G, 1 if residual else L, 1, H), dtype=torch.float32, device=dev)
    plan = M.RoutePlan.allocate(1, E, k, device=dev)
    ws = M.alloc_ffn_workspace(1, k, H, I, M.MOE_PATH_DECODE, device=dev)

    stream = torch.cuda.Stream(device=dev)

    def step(g):
        # one launch per layer: routing (top-k, softmax, histogram,
        # permutation), slot lookup, gate/up + SwiGLU, down + combine
        for l in range(L):
            M.moe_decode_layer(pool, l, lg_d[g, l], x_d[g, l], plan, slot_of, out_d[g, 0 if residual else l], ws,
                               stream=stream, accumulate=residual)

    # one CUDA graph per step (each step has its own inputs)
    graphs = []
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step(0)  # eager once before capture
    stream.synchronize()
    out_d.zero_()  # every graph below runs once: a residual row starts at zero
    for g in range(G):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(g)
        graphs.append(gr)
    torch.cuda.synchronize()

    for g in range(args.warmup):
        graphs[g].replay()
    torch.cuda.synchronize()

    import torch.distributed as dist

    def barrier():
        if world > 1:
            dist.barrier()

    clocks = Clocks(torch.cuda.current_device())
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for g in range(args.warmup, G):
            graphs[g].replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    # per-launch duration: the timed steps are back-to-back launches of the
    # decode kernel on this stream, so step time / launches per step
    ffn_ms = [elapsed_ms / args.steps / L]
    route_ms = [0.0]

    # e2e through the public API, host buffers, copies inside the timed region
    lg_pin = lg_h.pin_memory()
    x_pin = x_h.pin_memory()
    n_out = 1 if residual else L
    out_pin = torch.empty((G, n_out, 1, H), dtype=torch.float32).pin_memory()
    res_in = torch.zeros((n_out, 1, H), dtype=torch.float32).pin_memory()  # the residual row as it arrives
    lg_stage = torch.empty((L, 1, E), dtype=torch.float32, device=dev)
    x_stage = torch.empty((L, 1, H), dtype=torch.bfloat16, device=dev)
    out_stage = torch.empty((n_out, 1, H), dtype=torch.float32, device=dev)

    def e2e_step(g):
        lg_stage.copy_(lg_pin[g], non_blocking=True)
        x_stage.copy_(x_pin[g], non_blocking=True)
        if residual:
            out_stage.copy_(res_in, non_blocking=True)
        for l in range(L):
            M.moe_decode_layer(pool, l, lg_stage[l], x_stage[l], plan, slot_of, out_stage[0 if residual else l], ws,
                               stream=stream, accumulate=residual)
        out_pin[g].copy_(out_stage, non_blocking=True)
        stream.synchronize()

    with torch.cuda.stream(stream):
        for g in range(args.warmup):
            e2e_step(g)
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for g in range(args.warmup, G):
            e2e_step(g)
        b.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = a.elapsed_time(b)
    # the graphed and eager runs produced the same outputs, up to the fp32
    # rounding order of the cross-CTA atomic sums
    ref_o = out_d[args.warmup:].double()
    rel = float((out_pin[args.warmup:].to(dev).double() - ref_o).norm() / ref_o.norm().clamp_min(1e-30))
    same = rel <= 1e-6

    res = dict(elapsed_ms=elapsed_ms, ffn_ms=ffn_ms, route_ms=route_ms, clocks=clk, e2e_ms=e2e_ms,
               h2d=(lg_pin[0].numel() * 4 + x_pin[0].numel() * 2 + (res_in.numel() * 4 if residual else 0)),
               d2h=out_pin[0].numel() * 4,
               e2e_matches_graph=same, expert_bytes=eb)
    pool.close()
    return res


def _pinned_link_peak(dev):
    """Pinned-host -> device copy rate on this machine, GB/s (the bound of the
    staging workloads): three 1 GiB cudaMemcpyAsync copies, CUDA events."""
    import torch

    probe = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    probe_d = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    probe_d.copy_(probe, non_blocking=True)
    torch.cuda.synchronize()
    a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for _ in range(3):
        probe_d.copy_(probe, non_blocking=True)
    b0.record()
    torch.cuda.synchronize()
    return 3 * (1 << 30) / (a0.elapsed_time(b0) / 1e3) / 1e9


def _store_link_rate(host, eb, dev, n=48):
    """Copy rate from the expert store itself, GB/s: ``n`` whole experts
    spread over the store, each one cudaMemcpyAsync into a device scratch
    buffer, CUDA events.  Beside the fresh 1 GiB buffer of
    ``_pinned_link_peak`` it shows whether the store's own pages copy
    slower (a large pinned allocation need not get large pages)."""
    import torch

    count = host.numel() // eb
    idx = np.linspace(0, count - 1, num=min(n, count)).astype(np.int64)
    scratch = torch.empty(eb, dtype=torch.uint8, device=dev)
    scratch.copy_(host[:eb], non_blocking=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in idx:
        scratch.copy_(host[int(i) * eb:(int(i) + 1) * eb], non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    return len(idx) * eb / (a.elapsed_time(b) / 1e3) / 1e9


def staged_prefill_leg(args, wl):
    """Prefill of one layer through a pool of ``--prefill-slots`` slots (fewer
    than the routed experts), every expert in pinned host memory: per step,
    routing on the GPU, then moe_prefill_staged (windows of unique experts
    staged on a copy stream while the previous window's grouped GEMMs run).
    Timed end to end on the host clock and by CUDA events on the compute
    stream: x and logits come from pinned host memory, out goes back there."""
    import time

    import torch

    import routed_expert_ffn_histogram_gb300 as M

    dev = torch.device("cuda", torch.cuda.current_device())
    E, k, H, I, T, Sl = wl.experts, wl.top_k, wl.hidden, wl.inter, wl.tokens, args.prefill_slots
    window = args.window or Sl // 2
    eb = M.moe_expert_bytes(H, I)
    host = torch.empty(E * eb, dtype=torch.uint8).pin_memory()
    for e, w in enumerate(S.layer_weights(wl, 0)):
        M.moe_pack_expert(w, H, I, host.data_ptr() + e * eb)
    slots = torch.empty(Sl * eb, dtype=torch.uint8, device=dev)
    pool = M.Pool(1, E, Sl, H, I, host_experts=host, dev_slots=slots, preload=False, policy=args.policy)
    link_peak = _pinned_link_peak(dev)
    store_rate = _store_link_rate(host, eb, dev)
    G = 2  # two distinct input batches, alternated
    lg_pin = [torch.from_numpy(S.logits(wl, 0, g)).pin_memory() for g in range(G)]
    x_pin = [torch.from_numpy(S.activations_bf16_bits(wl, 0, g).view(np.int16)).view(torch.bfloat16).pin_memory()
             for g in range(G)]
    out_pin = torch.empty((T, H), dtype=torch.float32).pin_memory()
    lg_d = torch.empty((T, E), dtype=torch.float32, device=dev)
    x_d = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    out_d = torch.empty((T, H), dtype=torch.float32, device=dev)
    plan = M.RoutePlan.allocate(T, E, k, counts_host=True, device=dev)
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_PREFILL, device=dev)
    compute = torch.cuda.Stream(device=dev)
    copy = torch.cuda.Stream(device=dev)

    def step(g):
        lg_d.copy_(lg_pin[g % G], non_blocking=True)
        x_d.copy_(x_pin[g % G], non_blocking=True)
        M.moe_route_plan(lg_d, k, plan, stream=compute)
        pool.prefill_staged(0, plan.counts_host, window, k, x_bf16=x_d, plan=plan, out=out_d, workspace=ws,
                            compute=compute, copy=copy)
        out_pin.copy_(out_d, non_blocking=True)

    with torch.cuda.stream(compute):
        for g in range(args.warmup):
            step(g)
        compute.synchronize()
        c0 = pool.counters()
        clk = Clocks(torch.cuda.current_device())
        clk.start()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record(compute)
        for g in range(args.steps):
            step(g)
        b.record(compute)
        compute.synchronize()
        wall = (time.perf_counter() - t0) / args.steps * 1e3
        clocks = clk.stop()
    c1 = pool.counters()
    ms = a.elapsed_time(b) / args.steps
    h2d = c1["h2d_bytes"] - c0["h2d_bytes"]
    link = h2d / (ms * args.steps / 1e3) / 1e9
    misses = c1["misses"] - c0["misses"]
    uniq = int((plan.counts_host.numpy() > 0).sum())
    line = {"metric": METRIC, "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "mxf8f6f4->f32", "data": "synthetic",
            "config": {"workload": wl.name + f"_staged_s{Sl}_w{window}", "hidden": H, "inter": I, "experts": E,
                       "top_k": k, "tokens": T, "slots_per_layer": Sl, "window": window, "policy": args.policy,
                       "timing": "end to end: x and logits from pinned host memory, out back to it, every step"},
            "roofline": {"kernel": "miss staging: cudaMemcpyAsync of packed experts from pinned host, "
                                   "overlapping the previous window's grouped GEMMs",
                         "bound": "host_link", "achieved": link, "peak": link_peak, "unit": "GB/s",
                         "frac": link / link_peak, "peak_kind": "pinned H2D copy measured in this run",
                         "store_copy_gbs": store_rate,
                         "traffic": None, "bytes_per_miss": h2d // max(1, misses)},
            "staging": {"unique_experts_per_step": uniq, "misses_per_step": misses / args.steps,
                        "hits": c1["hits"] - c0["hits"], "events_per_step": (c1["events"] - c0["events"]) / args.steps,
                        "h2d_bytes_per_step": h2d / args.steps, "host_ms_per_step": wall},
            # per step: routing (top-k and scatter passes), quantisation, two GEMMs per window
            "gpu_launches": args.steps * (2 + 1 + 2 * ((uniq + window - 1) // window)),
            "e2e": {"value": T / (ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": lg_pin[0].numel() * 4 + x_pin[0].numel() * 2 + h2d / args.steps,
                    "d2h_bytes_per_step": out_pin.numel() * 4},
            "clocks": clocks}
    print(json.dumps(line))


def offload_leg(args, wl):
    """The GPT-OSS-shaped decode with a small GPU pool (8 of 32 slots per
    layer, LRU, skewed routing) and every expert in pinned host memory: per
    layer, routing on the GPU, the routed experts' counts to the host, the
    slot lookup and the copies of missed experts from pinned host memory on
    a copy stream, then the decode FFN.  Timed end to end: each step's
    logits and activations come from pinned host memory and its outputs go
    back there."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    dev = torch.device("cuda", torch.cuda.current_device())
    L = wl.layers if args.layers is None else min(args.layers, wl.layers)
    E, k, H, I, Sl = wl.experts, wl.top_k, wl.hidden, wl.inter, wl.slots
    eb = M.moe_expert_bytes(H, I)
    wsrc = S.WORKLOADS[wl.weight_wid]
    host = torch.empty(L * E * eb, dtype=torch.uint8).pin_memory()
    for l in range(L):
        for e, w in enumerate(S.layer_weights(wsrc, l)):
            M.moe_pack_expert(w, H, I, host.data_ptr() + (l * E + e) * eb)
    slots = torch.empty(L * Sl * eb, dtype=torch.uint8, device=dev)
    pool = M.Pool(L, E, Sl, H, I, host_experts=host, dev_slots=slots, preload=False, policy=args.policy,
                  stage_parts=args.stage_parts)

    link_peak = _pinned_link_peak(dev)
    store_rate = _store_link_rate(host, eb, dev)

    G = args.warmup + args.steps
    lg_pin = torch.from_numpy(np.stack([np.stack([S.logits(wl, l, g % wl.steps) for l in range(L)])
                                        for g in range(G)])).pin_memory()
    x_pin = torch.from_numpy(np.stack([np.stack([S.activations_bf16_bits(wl, l, g % wl.steps) for l in range(L)])
                                       for g in range(G)]).view(np.int16)).view(torch.bfloat16).pin_memory()
    out_pin = torch.empty((G, L, 1, H), dtype=torch.float32).pin_memory()
    lg_d = torch.empty((L, 1, E), dtype=torch.float32, device=dev)
    x_d = torch.empty((L, 1, H), dtype=torch.bfloat16, device=dev)
    out_d = torch.empty((L, 1, H), dtype=torch.float32, device=dev)
    plan = M.RoutePlan.allocate(1, E, k, counts_host=True, device=dev)
    slot_of = torch.empty(E, dtype=torch.int32, device=dev)
    ws = M.alloc_ffn_workspace(1, k, H, I, M.MOE_PATH_DECODE, device=dev)
    compute = torch.cuda.Stream(device=dev)
    copy = torch.cuda.Stream(device=dev)

    def step(g):
        lg_d.copy_(lg_pin[g], non_blocking=True)
        x_d.copy_(x_pin[g], non_blocking=True)
        for l in range(L):
            M.moe_route_plan(lg_d[l], k, plan, stream=compute)
            rc = pool.stage(l, plan.counts_host, slot_of, compute=compute, copy=copy)
            if rc != M.MOE_OK:
                raise RuntimeError(f"stage failed: {rc}")
            if args.prefetch:
                # the next layer's likely experts, copied while this layer computes
                pool.prefetch((l + 1) % L, args.prefetch, compute=compute, copy=copy)
            M.moe_expert_ffn(pool, l, x_d[l], plan, slot_of, out_d[l], ws, path=M.MOE_PATH_DECODE, stream=compute)
        out_pin[g].copy_(out_d, non_blocking=True)

    with torch.cuda.stream(compute):
        for g in range(args.warmup):
            step(g)
        compute.synchronize()
        c0 = pool.counters()
        clk = Clocks(torch.cuda.current_device())
        clk.start()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(compute)
        for g in range(args.warmup, G):
            step(g)
        b.record(compute)
        compute.synchronize()
        clocks = clk.stop()
    c1 = pool.counters()
    ms = a.elapsed_time(b) / args.steps
    h2d = c1["h2d_bytes"] - c0["h2d_bytes"]
    link = h2d / (ms * args.steps / 1e3) / 1e9
    line = {"metric": METRIC, "value": 1e3 / ms, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "layers": L, "hidden": H, "inter": I, "experts": E, "top_k": k,
                       "slots_per_layer": Sl, "routing_bias": wl.bias_c, "tokens_per_step": 1,
                       "timing": "end to end: inputs from and outputs to pinned host memory every step"},
            "roofline": {"kernel": "miss staging: cudaMemcpyAsync of packed experts from pinned host",
                         "bound": "host_link", "achieved": link, "peak": link_peak, "unit": "GB/s",
                         "frac": link / link_peak, "peak_kind": "pinned H2D copy measured in this run",
                         "store_copy_gbs": store_rate,
                         "traffic": None, "bytes_per_load": (c1["h2d_bytes"] - c0["h2d_bytes"]) //
                                                           max(1, c1["misses"] - c0["misses"] + c1["prefetches"] -
                                                               c0["prefetches"])},
            "offload": {"policy": args.policy, "stage_parts": args.stage_parts, "prefetch": args.prefetch,
                        "prefetches": c1["prefetches"] - c0["prefetches"],
                        "prefetch_hits": c1["prefetch_hits"] - c0["prefetch_hits"],
                        "hits": c1["hits"] - c0["hits"], "misses": c1["misses"] - c0["misses"],
                        "evictions": c1["evictions"] - c0["evictions"], "h2d_bytes": h2d,
                        "misses_per_step": (c1["misses"] - c0["misses"]) / args.steps},
            "e2e": {"value": 1e3 / ms, "unit": "tokens/s",
                    "h2d_bytes_per_step": (lg_pin[0].numel() * 4 + x_pin[0].numel() * 2) + h2d / args.steps,
                    "d2h_bytes_per_step": out_pin[0].numel() * 4},
            "gpu_launches": args.steps * L * 2,
            "clocks": clocks}
    if args.policy_sweep:
        line["policy_sweep"] = policy_sweep(wl, L, dev)
    print(json.dumps(line))


def policy_sweep(wl, L, dev):
    """Every (step, layer) routing event of the offload workload, routed on
    the GPU once, replayed through a policy-only pool (no copies) for each
    eviction policy: hits and misses over the whole stream, cold start."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    E, k = wl.experts, wl.top_k
    plan = M.RoutePlan.allocate(1, E, k, counts_host=True, device=dev)
    stream = torch.cuda.Stream(device=dev)
    events = []
    with torch.cuda.stream(stream):
        for step in range(wl.steps):
            lg = torch.from_numpy(np.stack([S.logits(wl, l, step) for l in range(L)])).to(dev)
            for l in range(L):
                M.moe_route_plan(lg[l], k, plan, stream=stream)
                stream.synchronize()
                events.append((l, plan.counts_host.numpy().copy()))
    out = {}
    for name in M.POLICIES:
        pool = M.Pool(L, E, wl.slots, wl.hidden, wl.inter, dry_run=True, policy=name)
        for l, c in events:
            pool.stage(l, c)
        c = pool.counters()
        out[name] = {"hits": c["hits"], "misses": c["misses"], "hit_rate": c["hits"] / max(1, c["hits"] + c["misses"]),
                     "misses_per_token": c["misses"] / wl.steps}
    return {"events": len(events), "steps": wl.steps, "layers": L, "policies": out}


def prefill_leg(args, wl):
    """One prefill layer call per step: routing + grouped tcgen05 expert FFN
    (the combine folded into the down GEMM's epilogue), graph-captured,
    inputs resident in HBM."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    dev = torch.device("cuda", torch.cuda.current_device())
    E, k, H, I, T = wl.experts, wl.top_k, wl.hidden, wl.inter, wl.tokens
    eb = M.moe_expert_bytes(H, I)
    host = torch.empty(E * eb, dtype=torch.uint8).pin_memory()
    for e, w in enumerate(S.layer_weights(wl, 0)):
        M.moe_pack_expert(w, H, I, host.data_ptr() + e * eb)
    slots = torch.empty(E * eb, dtype=torch.uint8, device=dev)
    pool = M.Pool(1, E, E, H, I, host_experts=host, dev_slots=slots, preload=True)
    slot_of = torch.arange(E, dtype=torch.int32, device=dev)
    G = 2  # two distinct input batches, alternated
    lg = [torch.from_numpy(S.logits(wl, 0, g)).to(dev) for g in range(G)]
    xb = [torch.from_numpy(S.activations_bf16_bits(wl, 0, g).view(np.int16)).to(dev).view(torch.bfloat16)
          for g in range(G)]
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    plans = [M.RoutePlan.allocate(T, E, k, device=dev) for _ in range(G)]
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_PREFILL, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    ext = dict(enable_timing=True)
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        ext["external"] = True
    except TypeError:
        pass
    ev = [(torch.cuda.Event(**ext), torch.cuda.Event(**ext), torch.cuda.Event(**ext)) for _ in range(G)]

    def step(g):
        e0, e1, e2 = ev[g]
        flush.fill_(g)  # larger than L2: every step starts from a cold L2
        e0.record(stream)
        M.moe_route_plan(lg[g], k, plans[g], stream=stream, with_counts_host=False)
        e1.record(stream)
        M.moe_expert_ffn(pool, 0, xb[g], plans[g], slot_of, out, ws, path=M.MOE_PATH_PREFILL, stream=stream,
                         accumulate=args.output == "residual")
        e2.record(stream)

    with torch.cuda.stream(stream):
        step(0)
    stream.synchronize()
    graphs = []
    for g in range(G):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(g)
        graphs.append(gr)
    for i in range(args.warmup):
        graphs[i % G].replay()
    torch.cuda.synchronize()
    route_ms, ffn_ms = [], []
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    total = 0.0
    for i in range(args.steps):
        graphs[i % G].replay()
        torch.cuda.synchronize()
        e0, e1, e2 = ev[i % G]
        route_ms.append(e0.elapsed_time(e1))
        ffn_ms.append(e1.elapsed_time(e2))
        total += e0.elapsed_time(e2)
    clk = clocks.stop()
    pool.close()
    return dict(step_ms=total / args.steps, route_ms=route_ms, ffn_ms=ffn_ms, clocks=clk)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-layers", type=int, default=4, help="layers per oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", type=int, default=1, choices=[1, 2, 3, 4],
                    help="1: GPT-OSS decode (default); 2: the same with an 8-slot offload pool; "
                         "3, 4: prefill layers (extra measurements)")
    ap.add_argument("--policy", default="lru", choices=["lru", "fifo", "lfu", "lfru", "slru"],
                    help="eviction policy of the offload pool (--workload 2)")
    ap.add_argument("--stage-parts", default="whole", choices=["whole", "decode"],
                    help="--workload 2: copy whole experts, or only what the decode kernel reads")
    ap.add_argument("--output", default="residual", choices=["residual", "overwrite"],
                    help="decode: each layer adds into the step's residual row (moe_decode_layer_acc) or "
                         "overwrites its own output (moe_decode_layer)")
    ap.add_argument("--prefetch", type=int, default=0,
                    help="workload 2: after each layer's staging, prefetch up to this many experts of the next layer")
    ap.add_argument("--prefill-slots", type=int, default=None,
                    help="workloads 3/4: run the layer through a pool of this many slots (moe_prefill_staged)")
    ap.add_argument("--window", type=int, default=None,
                    help="with --prefill-slots: unique experts per staging window (default slots // 2)")
    ap.add_argument("--policy-sweep", action="store_true",
                    help="with --workload 2: also replay the whole routing stream under every policy")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers (smaller case for profiler captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = _dist()
    wl = S.WORKLOADS[args.workload]
    if args.workload == 2:
        import torch

        torch.cuda.set_device(0)
        from routed_expert_ffn_histogram_gb300 import build as B

        B.build()
        offload_leg(args, wl)
        return
    if args.workload in (3, 4):
        import torch

        torch.cuda.set_device(0)
        from routed_expert_ffn_histogram_gb300 import build as B

        B.build()
        if args.prefill_slots:
            staged_prefill_leg(args, wl)
            return
        res = prefill_leg(args, wl)
        flops = 6.0 * wl.hidden * wl.inter * wl.tokens * wl.top_k
        ffn_s = statistics.median(res["ffn_ms"]) / 1e3
        _, bf16_peak, peak_kind = _peaks()
        tc_peak = bf16_peak * 2.0  # kind::mxf8f6f4 issues at the FP8 rate: 2x the measured bf16 rate
        achieved = flops / ffn_s / 1e12
        line = {"metric": METRIC, "value": wl.tokens / (res["step_ms"] / 1e3), "unit": "tokens/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["step_ms"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxf8f6f4->f32",
                "data": "synthetic",
                "config": {"workload": wl.name, "hidden": wl.hidden, "inter": wl.inter, "experts": wl.experts,
                           "top_k": wl.top_k, "tokens": wl.tokens, "l2": "256 MB flush before every step",
                           "output": ("added into a residual stream (MOE_FFN_ACCUMULATE)" if args.output == "residual"
                                      else "overwritten (out zeroed, then the combine adds into it)")},
                "roofline": {"kernel": "prefill expert FFN (MXFP8 quant, gate/up GEMM, down GEMM with the combine in its epilogue)",
                             "bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                             "frac": achieved / tc_peak, "peak_kind": peak_kind + " bf16 x 2 (FP8-class rate)",
                             "traffic": NCU_TRAFFIC.get("grouped_gemm_tc_kernel/" + wl.name),
                             "traffic_scope": "DRAM bytes of the two GEMM launches of one layer",
                             "algorithmic_flops_per_launch": flops,
                             "avg_launch_us": ffn_s * 1e6},
                "kernels_us": {"route_plan": statistics.median(res["route_ms"]) * 1e3,
                               "expert_ffn": ffn_s * 1e6},
                "clocks": res["clocks"]}
        print(json.dumps(line))
        return
    if args.layers:
        import dataclasses

        wl = dataclasses.replace(wl, layers=min(args.layers, wl.layers))
    hbm_peak, _, peak_kind = _peaks()
    workload = {"workload": wl.name, "layers": wl.layers, "hidden": wl.hidden, "inter": wl.inter,
                "experts": wl.experts, "top_k": wl.top_k, "tokens_per_step": 1,
                "resident_experts": wl.layers * wl.experts,
                "l2": "inputs larger than L2: each step reads 96 distinct experts (1.27 GB) of a 10.2 GB set",
                "output": ("each layer adds into the step's residual row (moe_decode_layer_acc)"
                           if args.output == "residual" else "each layer overwrites its own output (moe_decode_layer)"),
                "parallelism": f"replicas{world}"}
    threads = os.cpu_count() or 1
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle

        oracle.build()
        tps, layers, times = oracle_leg(wl, args.warmup + args.steps, args.cpu_layers, threads)
        timed = times[args.warmup:]
        per_token = statistics.median(timed) * wl.layers / len(layers)
        v = 1.0 / per_token
        sample = f"{len(layers)} of {wl.layers} layers per step (layers {layers}), scaled to {wl.layers} layers"
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 0,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_token * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic", "config": workload,
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from routed_expert_ffn_histogram_gb300 import build as B

    B.build()
    res = gpu_leg(args, wl, rank, world)
    ms = res["elapsed_ms"] / args.steps
    e2e_ms = res["e2e_ms"] / args.steps
    ms, e2e_ms = reduce_max_over_ranks([ms, e2e_ms], world, device="cuda")
    if rank != 0:
        return
    value = world * 1e3 / ms
    layer_bytes = wl.top_k * 3 * (wl.hidden * wl.inter // 2 + wl.hidden * wl.inter // 32)
    ffn_avg_s = statistics.mean(res["ffn_ms"]) / 1e3
    achieved = layer_bytes / ffn_avg_s / 1e9
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": workload,
            "formats": "weights MXFP4 (E2M1 + E8M0 per 32), activations bf16, fp32 accumulation",
            "roofline": {"kernel": "decode_fused_kernel: one launch per layer (routing, gate/up+SwiGLU, "
                                   "down+combine)",
                         "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "peak_kind": peak_kind,
                         "traffic": NCU_TRAFFIC["decode_fused_kernel"],
                         "algorithmic_bytes_per_launch": layer_bytes,
                         "avg_launch_us": ffn_avg_s * 1e6},
            "kernels_us": {"decode_layer": ffn_avg_s * 1e6},
            "e2e": {"value": world * 1e3 / e2e_ms, "unit": "tokens/s", "h2d_bytes_per_step": res["h2d"],
                    "d2h_bytes_per_step": res["d2h"], "matches_graph_outputs": res["e2e_matches_graph"]},
            "gpu_launches": args.steps * wl.layers,
            "clocks": res["clocks"]}
    if not args.no_cpu_baseline:
        import oracle

        oracle.build()
        tps, layers, times = oracle_leg(wl, 1, args.cpu_layers, threads)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": f"1 decode step, {len(layers)} of {wl.layers} layers "
                                          f"({layers}), scaled to {wl.layers} layers"}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
