#!/usr/bin/env python
"""Benchmark of the routed-expert FFN layer on GB300.

Headline (``value``): GPT-OSS-20B-shaped decode with every expert resident --
24 stacked MoE layers (hidden 2880, expert intermediate 2880, 32 experts,
top-4), one token per step, 768 distinct MXFP4 experts (10.2 GB) in the GPU
slot pool.  One step = one token through all 24 layers: routing (top-k,
softmax, histogram, permutation), the slot lookup, gate/up + SwiGLU, down,
and the weighted combine.

The same JSON line (one GPU) also carries the rest of the metric:
  prefill  the 3072-token GPT-OSS-shaped and the 16384-token
           Qwen-30B-A3B-shaped prefill layers (tcgen05 grouped GEMM), with
           TFLOP/s against the measured rate of the MMA instruction they issue;
  offload  the GPT-OSS-shaped decode through an 8-of-32-slot pool per layer
           (LRU, skewed routing), end to end with the misses copied from
           pinned host memory, against the pinned copy rate of this machine;
  peaks    those measured denominators.
Each part has its roofline, an end-to-end figure through the C ABI from
pinned host buffers, and the CPU oracle timed on a bounded sample.

``--impl reference`` times the CPU oracle on the host cores instead.
``--workload 2|3|4`` prints the line of one of the other workloads alone.

Multi-GPU: the layer does not shard in this form (one token's four experts);
``--gpus N`` under torchrun runs N independent decode replicas and reports
the sum (the prefill and offload parts are measured on one GPU only).
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
    "decode_fused_kernel": 54_206_208 + 7_936,
    # one layer of the 24-layer GGUF leg (a launch after 40 others)
    "gguf_fused_kernel/q4_k": 21_341_440 + 0,
    "gguf_fused_kernel/q8_0": 40_212_736 + 2_304,
    # gate/up launch + down launch of one 3072-token GPT-OSS-shaped layer
    "grouped_gemm_tc_kernel/gptoss20b_prefill_t3072": (320_126_976 + 31_258_624) + (234_308_096 + 31_640_832),
}

# Dense tensor-core rates of GB300 in the published ratios (bf16 : fp8 : fp4
# = 2.25 : 4.5 : 13.5 PFLOP/s): the MXFP4 (kind::mxf4) rate is the measured
# bf16 rate times 6.
FP4_OVER_BF16 = 13.5 / 2.25


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling (every ``interval_ms``) while a region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, interval_ms: int = 50):
        self.idx = device_index
        self.interval = interval_ms
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
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
                "reasons": sorted(reasons), "samples": len(rows), "interval_ms": self.interval,
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


def _events(n=2):
    import torch

    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _graph_event():
    """A timing event that can be recorded inside a captured CUDA graph and
    timed after a replay (an external event where torch offers it)."""
    import torch

    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


def _soak(fn, seconds: float):
    """Run ``fn`` (enqueues GPU work) back to back for about ``seconds``."""
    import torch

    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < seconds:
        fn(n)
        n += 1
        if n % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return n, time.perf_counter() - t0


# --------------------------------------------------------------------------
# oracle legs (CPU baseline / reference arm)
# --------------------------------------------------------------------------

def _oracle_decode_sample(wl, step, layers, weights_cache, threads):
    """Time the oracle on ``layers`` of one decode step; returns seconds."""
    import oracle

    t0 = time.perf_counter()
    for l in layers:
        lg = S.logits(wl, l, step)
        ids, w = oracle.route(lg, wl.top_k)
        oracle.hist_perm(ids, wl.experts)
        x = S.activations_bf16_bits(wl, l, step)
        oracle.layer(x, ids, w, weights_cache[l], prefill=False, threads=threads)
    return time.perf_counter() - t0


def _sample_layers(wl, n):
    return list(range(0, wl.layers, max(1, wl.layers // n)))[:n]


def cpu_decode_baseline(wl, layers_per_sample, threads, steps=1):
    """Oracle tokens/s on ``steps`` decode steps, ``layers_per_sample`` of
    the 24 layers each, scaled to the whole stack."""
    layers = _sample_layers(wl, layers_per_sample)
    cache = {l: S.stack_experts(S.layer_weights(wl, l)) for l in layers}
    times = [_oracle_decode_sample(wl, s, layers, cache, threads) for s in range(steps)]
    per_token = statistics.median(times) * wl.layers / len(layers)
    return {"value": 1.0 / per_token, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{steps} decode step(s), {len(layers)} of {wl.layers} layers ({layers}), "
                      f"scaled to {wl.layers} layers"}


def cpu_offload_baseline(wl, layers_per_sample, threads):
    """Oracle tokens/s of the offload workload: the layers of one step as in
    the resident decode, plus the oracle's slot-pool simulation of every
    layer's event of that step (the oracle keeps all experts in host memory,
    so it has no copies)."""
    import oracle

    layers = _sample_layers(wl, layers_per_sample)
    wsrc = S.WORKLOADS[wl.weight_wid]
    cache = {l: S.stack_experts(S.layer_weights(wsrc, l)) for l in layers}
    t0 = time.perf_counter()
    pools = [oracle.LRUPool(wl.slots, wl.experts) for _ in range(wl.layers)]
    for l in range(wl.layers):
        ids, _ = oracle.route(S.logits(wl, l, 0), wl.top_k)
        counts, _, _, _ = oracle.hist_perm(ids, wl.experts)
        pools[l].step(counts)
    t_pool = time.perf_counter() - t0
    t_layers = _oracle_decode_sample(wl, 0, layers, cache, threads)
    per_token = t_pool + t_layers * wl.layers / len(layers)
    return {"value": 1.0 / per_token, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"1 step: the LRU simulation of all {wl.layers} layers' events and {len(layers)} of "
                      f"{wl.layers} layers' expert FFN ({layers}), scaled to {wl.layers} layers"}


def cpu_prefill_baseline(wl, tokens, threads):
    """Oracle tokens/s of a prefill layer on the first ``tokens`` tokens
    (routing of those tokens, then the layer on the MXFP8 path)."""
    import oracle

    ws = S.stack_experts(S.layer_weights(wl, 0))
    lg = S.logits(wl, 0, 0)[:tokens]
    x = S.activations_bf16_bits(wl, 0, 0)[:tokens]
    t0 = time.perf_counter()
    ids, w = oracle.route(lg, wl.top_k)
    oracle.hist_perm(ids, wl.experts)
    oracle.layer(x, ids, w, ws, prefill=True, threads=threads)
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"the first {tokens} of {wl.tokens} tokens of the layer (routing + MXFP8 expert FFN)"}


# --------------------------------------------------------------------------
# GPU legs
# --------------------------------------------------------------------------

def build_host_store(M, wl, layers):
    """Pinned host tensor [layers][E][expert_bytes] of packed experts."""
    import torch

    E, H, I = wl.experts, wl.hidden, wl.inter
    eb = M.moe_expert_bytes(H, I)
    host = torch.empty(layers * E * eb, dtype=torch.uint8).pin_memory()
    src = S.WORKLOADS[wl.weight_wid]
    for l in range(layers):
        for e, w in enumerate(S.layer_weights(src, l)):
            M.moe_pack_expert(w, H, I, host.data_ptr() + (l * E + e) * eb)
    return host


def gpu_decode_leg(args, wl, host, rank, world):
    """The headline: per layer one moe_decode_layer(_acc) launch, each step's
    24 launches captured in a CUDA graph of their own."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    dev = torch.device("cuda", torch.cuda.current_device())
    L, E, k, H, I = wl.layers, wl.experts, wl.top_k, wl.hidden, wl.inter
    eb = M.moe_expert_bytes(H, I)
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

    def replay(n):
        with torch.cuda.stream(stream):
            graphs[args.warmup + n % args.steps].replay()

    # clocks are sampled over a soak of the same step graphs that encloses
    # the timed region (about a second in all); the K timed steps start
    # from outputs cleared after the first soak
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    soak_n, soak_s = _soak(replay, args.soak / 2)
    out_d.zero_()
    t_start, t_end = _events()
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for g in range(args.warmup, G):
            graphs[g].replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    graph_out = out_d.clone()
    soak_n2, soak_s2 = _soak(replay, args.soak / 2)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    # the same K steps once more, each step between its own pair of events:
    # median and coefficient of variation of the step time
    step_ev = [_events() for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for n, g in enumerate(range(args.warmup, G)):
            step_ev[n][0].record(stream)
            graphs[g].replay()
            step_ev[n][1].record(stream)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]

    # e2e through the public API, host buffers, copies inside the timed region:
    # every step's logits, activations and residual row go up from pinned
    # memory and its row comes back to pinned memory.  Two sets of staging
    # buffers and two streams: step g + 1's inputs upload and step g's row
    # reads back while step g computes (the prefill e2e's arrangement); the
    # step's 24 C-ABI calls on a buffer set are captured once per set and
    # replayed.  Host clock over the whole run, ending after the last row
    # has reached host memory.
    lg_pin = lg_h.pin_memory()
    x_pin = x_h.pin_memory()
    n_out = 1 if residual else L
    out_pin = torch.empty((G, n_out, 1, H), dtype=torch.float32).pin_memory()
    res_in = torch.zeros((n_out, 1, H), dtype=torch.float32).pin_memory()  # the residual row as it arrives
    lg_stage = [torch.empty((L, 1, E), dtype=torch.float32, device=dev) for _ in range(2)]
    x_stage = [torch.empty((L, 1, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    out_stage = [torch.empty((n_out, 1, H), dtype=torch.float32, device=dev) for _ in range(2)]
    compute = torch.cuda.Stream(device=dev)
    copy = torch.cuda.Stream(device=dev)

    def layer_calls(b):
        for l in range(L):
            M.moe_decode_layer(pool, l, lg_stage[b][l], x_stage[b][l], plan, slot_of,
                               out_stage[b][0 if residual else l], ws, stream=compute, accumulate=residual)

    calls = []
    for b in range(2):
        with torch.cuda.stream(compute):
            layer_calls(b)
        compute.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=compute):
            layer_calls(b)
        calls.append(gr)
    up_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def upload(g):
        b = g % 2
        with torch.cuda.stream(copy):
            if g >= 2:
                copy.wait_event(comp_done[b])   # step g - 2 no longer reads buffer set b
            lg_stage[b].copy_(lg_pin[g], non_blocking=True)
            x_stage[b].copy_(x_pin[g], non_blocking=True)
            if residual:
                out_stage[b].copy_(res_in, non_blocking=True)
            up_done[b].record(copy)

    def run(g):
        b = g % 2
        with torch.cuda.stream(compute):
            compute.wait_event(up_done[b])
            calls[b].replay()
            comp_done[b].record(compute)
        with torch.cuda.stream(copy):
            copy.wait_event(comp_done[b])
            out_pin[g].copy_(out_stage[b], non_blocking=True)

    def e2e_run(g0, g1):
        upload(g0)
        for g in range(g0, g1):
            if g + 1 < g1:
                upload(g + 1)
            run(g)
        torch.cuda.synchronize()

    e2e_run(0, args.warmup)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e2e_run(args.warmup, G)
    e2e_ms = (time.perf_counter() - t0) * 1e3
    barrier()
    # the step graphs and the replayed C-ABI calls produced the same outputs,
    # up to the fp32 rounding order of the cross-CTA atomic sums
    ref_o = graph_out[args.warmup:].double()
    rel = float((out_pin[args.warmup:].to(dev).double() - ref_o).norm() / ref_o.norm().clamp_min(1e-30))
    res = dict(elapsed_ms=elapsed_ms, clocks=clk, e2e_ms=e2e_ms, step_ms=step_ms,
               soak={"steps": soak_n + soak_n2, "seconds": soak_s + soak_s2},
               h2d=(lg_pin[0].numel() * 4 + x_pin[0].numel() * 2 + (res_in.numel() * 4 if residual else 0)),
               d2h=out_pin[0].numel() * 4, e2e_matches_graph=rel <= 1e-6, expert_bytes=eb)
    pool.close()
    del slots
    torch.cuda.empty_cache()
    return res


def _pinned_link_peak(dev):
    """Pinned-host -> device copy rate on this machine, GB/s (the bound of the
    staging workloads): three 1 GiB cudaMemcpyAsync copies, CUDA events."""
    import torch

    probe = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    probe_d = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    probe_d.copy_(probe, non_blocking=True)
    torch.cuda.synchronize()
    a0, b0 = _events()
    a0.record()
    for _ in range(3):
        probe_d.copy_(probe, non_blocking=True)
    b0.record()
    torch.cuda.synchronize()
    return 3 * (1 << 30) / (a0.elapsed_time(b0) / 1e3) / 1e9


def _store_warm_pass(host, eb, dev):
    """Every expert of the store copied once into a device scratch buffer;
    returns the pass's rate, GB/s (host clock)."""
    import torch

    scratch = torch.empty(eb, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(host.numel() // eb):
        scratch.copy_(host[i * eb:(i + 1) * eb], non_blocking=True)
    torch.cuda.synchronize()
    return host.numel() / (time.perf_counter() - t0) / 1e9


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
    a, b = _events()
    a.record()
    for i in idx:
        scratch.copy_(host[int(i) * eb:(int(i) + 1) * eb], non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    return len(idx) * eb / (a.elapsed_time(b) / 1e3) / 1e9


def measure_mma_peak(dev, seconds=1.0):
    """Rate of tcgen05.mma.kind::mxf8f6f4 (M128 N256 K32, E4M3 x E2M1, E8M0
    block scales), the instruction of the prefill GEMMs: the library's probe
    (one CTA per SM issuing back-to-back MMAs on operands resident in shared
    memory) timed with CUDA events.  Burst: best of five 4096-stage launches;
    sustained: launches back to back for about ``seconds``."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stages = 4096
    ctas = M.moe_probe_mxf8f6f4(stages, status)  # warm-up
    torch.cuda.synchronize()
    flops = ctas * stages * 4 * 2.0 * 128 * 256 * 32
    best = 0.0
    for _ in range(5):
        a, b = _events()
        a.record()
        M.moe_probe_mxf8f6f4(stages, status)
        b.record()
        torch.cuda.synchronize()
        best = max(best, flops / (a.elapsed_time(b) / 1e3) / 1e12)
    n = max(1, int(seconds / (flops / max(best, 1.0) / 1e12)))
    a, b = _events()
    a.record()
    for _ in range(n):
        M.moe_probe_mxf8f6f4(stages, status)
    b.record()
    torch.cuda.synchronize()
    sustained = n * flops / (a.elapsed_time(b) / 1e3) / 1e12
    if int(status.item()) != 0:
        raise RuntimeError(f"tensor-core probe wait ran out (status {int(status.item())})")
    return {"burst_tflops": best, "sustained_tflops": sustained, "ctas": ctas,
            "how": "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale M128 N256 K32 back to back, operands in "
                   "shared memory, one CTA per SM, CUDA events (moe_probe_mxf8f6f4)"}


def offload_obj(args, wl, host):
    """The GPT-OSS-shaped decode with a small GPU pool (8 of 32 slots per
    layer, skewed routing) and every expert in pinned host memory: per
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
    slots = torch.empty(L * Sl * eb, dtype=torch.uint8, device=dev)
    pool = M.Pool(L, E, Sl, H, I, host_experts=host, dev_slots=slots, preload=False, policy=args.policy,
                  stage_parts=args.stage_parts)
    # One pass over the whole store first (every expert copied once): the
    # first device reads of a store the CPU has just packed run at a
    # fraction of the link rate, a one-time cost of loading that a server
    # pays before it serves, not a per-token cost.
    warm_gbs = _store_warm_pass(host, eb, dev)
    # the host copy rates right before and after the timed region: a fresh
    # 1 GiB pinned buffer and whole experts out of the store itself (the
    # store's rate has been seen to vary between boxes and runs)
    rates = {"pinned_1gib_before": _pinned_link_peak(dev), "store_before": _store_link_rate(host, eb, dev),
             "store_warm_pass": warm_gbs}
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
        a, b = _events()
        t0 = time.perf_counter()
        a.record(compute)
        for g in range(args.warmup, G):
            step(g)
        b.record(compute)
        compute.synchronize()
        wall_ms = (time.perf_counter() - t0) / args.steps * 1e3
        clocks = clk.stop()
    c1 = pool.counters()
    pool.close()
    dv = _offload_device_planned(args, wl, host, slots, lg_pin, x_pin, dev, L)
    rates.update(pinned_1gib_after=_pinned_link_peak(dev), store_after=_store_link_rate(host, eb, dev))
    link_peak = max(rates["pinned_1gib_before"], rates["pinned_1gib_after"])
    store_rate = min(rates["store_before"], rates["store_after"])
    ms_host = a.elapsed_time(b) / args.steps
    h2d_host = c1["h2d_bytes"] - c0["h2d_bytes"]
    host_planned = {"value": 1e3 / ms_host, "unit": "tokens/s", "ms_per_step": ms_host, "host_ms_per_step": wall_ms,
                    "link_gbs": h2d_host / (ms_host * args.steps / 1e3) / 1e9,
                    "misses": c1["misses"] - c0["misses"], "hits": c1["hits"] - c0["hits"],
                    "how": "per layer: routing, counts to pinned host memory, host waits for them, plans "
                           "(moe_pool_stage), one cudaMemcpyAsync per staged part of each miss on a copy stream, "
                           "the FFN after an event on it; eager calls"}
    ms, c0, c1, clocks = dv["ms"], dv["c0"], dv["c1"], dv["clocks"]
    h2d = c1["h2d_bytes"] - c0["h2d_bytes"]
    link = h2d / (ms * args.steps / 1e3) / 1e9
    misses = c1["misses"] - c0["misses"]
    ref_o = out_pin.double()
    out_rel = float((dv["out"].double() - ref_o).norm() / ref_o.norm().clamp_min(1e-30))
    obj = {"workload": wl.name, "value": 1e3 / ms, "unit": "tokens/s", "ms_per_step": ms,
           "host_planned": host_planned, "same_events_as_host_planned": (misses, c1["hits"] - c0["hits"]) == (
               host_planned["misses"], host_planned["hits"]),
           "outputs_vs_host_planned_rel_l2": out_rel,
           "config": {"layers": L, "hidden": H, "inter": I, "experts": E, "top_k": k, "slots_per_layer": Sl,
                      "routing_bias": wl.bias_c, "policy": args.policy, "stage_parts": args.stage_parts,
                      "prefetch": args.prefetch, "tokens_per_step": 1,
                      "timing": "end to end through the C ABI: each step's logits and activations from pinned "
                                "host memory, per layer routing and the staging event planned on the GPU in one "
                                "launch (moe_pool_route_stage_device), misses copied by the SMs from the mapped "
                                "pinned expert "
                                "store on a second stream while the FFN of the event's hits runs, the FFN of the "
                                "loaded experts on that stream right behind the copy, outputs back to pinned host "
                                "memory; one CUDA graph "
                                "per step (24 x (routing + plan, (copy, loads' FFN) | hits' FFN) plus the input and "
                                "output copies), CUDA events"},
           "roofline": {"kernel": "miss staging: SM copy of packed experts out of mapped pinned host memory",
                        "bound": "host_link", "achieved": link, "peak": link_peak, "unit": "GB/s",
                        "frac": link / link_peak, "peak_kind": "pinned H2D copy of a fresh 1 GiB buffer, best of "
                                                               "the measurements just before and after",
                        "store_copy_gbs": store_rate, "frac_of_store_rate": link / store_rate,
                        "copy_rates_gbs": rates, "traffic": None,
                        "bytes_per_load": h2d // max(1, misses + c1["prefetches"] - c0["prefetches"])},
           "staging": {"hits": c1["hits"] - c0["hits"], "misses": misses, "evictions": c1["evictions"] - c0["evictions"],
                       "misses_per_step": misses / args.steps, "h2d_bytes": h2d,
                       "prefetches": c1["prefetches"] - c0["prefetches"],
                       "prefetch_hits": c1["prefetch_hits"] - c0["prefetch_hits"],
                       "hit_rate": (c1["hits"] - c0["hits"]) / max(1, c1["hits"] - c0["hits"] + misses)},
           "e2e": {"value": 1e3 / ms, "unit": "tokens/s",
                   "h2d_bytes_per_step": (lg_pin[0].numel() * 4 + x_pin[0].numel() * 2) + h2d / args.steps,
                   "d2h_bytes_per_step": out_pin[0].numel() * 4},
           "gpu_launches": args.steps * L * dv["launches_per_layer"],
           "clocks": clocks}
    del slots
    torch.cuda.empty_cache()
    return obj


def _offload_device_planned(args, wl, host, slots, lg_pin, x_pin, dev, L, split=True):
    """The offload decode with device-planned staging: the pool's state in
    device memory; per layer routing + planning (one launch,
    moe_pool_route_stage_device), then the SM copy of the misses
    on a second stream while the FFN of the event's hits runs, the FFN of
    the loaded experts on that stream right behind the copy (both adding
    into the zeroed output), and the compute stream joined to it; each step
    (with its input and output copies) one CUDA graph.  Same events as the
    host-planned run (same routing stream, same policy, a fresh pool)."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    E, k, H, I, Sl = wl.experts, wl.top_k, wl.hidden, wl.inter, wl.slots
    G = args.warmup + args.steps
    pool = M.Pool(L, E, Sl, H, I, host_experts=host, dev_slots=slots, preload=False, policy=args.policy,
                  stage_parts=args.stage_parts)
    stream = torch.cuda.Stream(device=dev)
    copy = torch.cuda.Stream(device=dev)
    maps = torch.empty((2, E), dtype=torch.int32, device=dev)
    state = torch.zeros(pool.device_state_bytes(), dtype=torch.uint8, device=dev)
    lg_d = torch.empty((L, 1, E), dtype=torch.float32, device=dev)
    x_d = torch.empty((L, 1, H), dtype=torch.bfloat16, device=dev)
    out_d = torch.empty((L, 1, H), dtype=torch.float32, device=dev)
    out_pin = torch.empty((G, L, 1, H), dtype=torch.float32).pin_memory()
    plan = M.RoutePlan.allocate(1, E, k, device=dev)
    slot_of = torch.empty(E, dtype=torch.int32, device=dev)
    ws = M.alloc_ffn_workspace(1, k, H, I, M.MOE_PATH_DECODE, device=dev)
    ws_loads = M.alloc_ffn_workspace(1, k, H, I, M.MOE_PATH_DECODE, device=dev)
    joined = [torch.cuda.Event() for _ in range(L)]
    pool.device_attach(state, stream=stream)

    def body(g):
        lg_d.copy_(lg_pin[g], non_blocking=True)
        x_d.copy_(x_pin[g], non_blocking=True)
        if split:
            out_d.zero_()
        for l in range(L):
            # routing and the staging event's planning in one launch
            if split:
                pool.route_stage_device(l, lg_d[l], k, plan, slot_of, split_dev=maps, stream=stream, copy=copy)
                # the hits' part beside the copy; the loads' part on the copy
                # stream right behind it; both add into the zeroed output
                M.moe_expert_ffn(pool, l, x_d[l], plan, maps[0], out_d[l], ws, path=M.MOE_PATH_DECODE,
                                 stream=stream, skip_absent=True, accumulate=True)
                M.moe_expert_ffn(pool, l, x_d[l], plan, maps[1], out_d[l], ws_loads, path=M.MOE_PATH_DECODE,
                                 stream=copy, skip_absent=True, accumulate=True)
                joined[l].record(copy)
                stream.wait_event(joined[l])
                pool.device_join(l, stream=stream)
            else:
                pool.route_stage_device(l, lg_d[l], k, plan, slot_of, stream=stream)
                M.moe_expert_ffn(pool, l, x_d[l], plan, slot_of, out_d[l], ws, path=M.MOE_PATH_DECODE,
                                 stream=stream)
        out_pin[g].copy_(out_d, non_blocking=True)

    graphs = []
    for g in range(G):
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=stream):
            body(g)
        graphs.append(cg)
    with torch.cuda.stream(stream):
        for g in range(args.warmup):
            graphs[g].replay()
    stream.synchronize()
    assert pool.device_detach(stream=stream) == M.MOE_OK
    c0 = pool.counters()
    pool.device_attach(state, stream=stream)
    clk = Clocks(torch.cuda.current_device())
    clk.start()
    a, b = _events()
    with torch.cuda.stream(stream):
        a.record(stream)
        for g in range(args.warmup, G):
            graphs[g].replay()
        b.record(stream)
    stream.synchronize()
    clocks = clk.stop()
    assert pool.device_detach(stream=stream) == M.MOE_OK
    c1 = pool.counters()
    pool.close()
    del graphs
    return {"ms": a.elapsed_time(b) / args.steps, "c0": c0, "c1": c1, "clocks": clocks,
            "launches_per_layer": 4 if split else 3, "out": out_pin}


def _prefill_setup(M, wl, dev):
    import torch

    E, H, I = wl.experts, wl.hidden, wl.inter
    eb = M.moe_expert_bytes(H, I)
    host = torch.empty(E * eb, dtype=torch.uint8).pin_memory()
    for e, w in enumerate(S.layer_weights(wl, 0)):
        M.moe_pack_expert(w, H, I, host.data_ptr() + e * eb)
    slots = torch.empty(E * eb, dtype=torch.uint8, device=dev)
    pool = M.Pool(1, E, E, H, I, host_experts=host, dev_slots=slots, preload=True)
    return host, slots, pool


def prefill_timing(args, wl, soak_s=0.0):
    """One prefill layer call per step: routing + grouped tcgen05 expert FFN
    (the combine folded into the down GEMM's epilogue), graph-captured,
    inputs resident in HBM, L2 flushed before every step.  Also the same
    layer end to end through the C ABI from pinned host buffers (two
    streams: step g + 1's inputs upload and step g - 1's output downloads
    while step g computes)."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    dev = torch.device("cuda", torch.cuda.current_device())
    E, k, H, I, T = wl.experts, wl.top_k, wl.hidden, wl.inter, wl.tokens
    host, slots, pool = _prefill_setup(M, wl, dev)
    slot_of = torch.arange(E, dtype=torch.int32, device=dev)
    G = 2  # two distinct input batches, alternated
    lg_h = [torch.from_numpy(S.logits(wl, 0, g)) for g in range(G)]
    x_h = [torch.from_numpy(S.activations_bf16_bits(wl, 0, g).view(np.int16)).view(torch.bfloat16) for g in range(G)]
    lg = [t.to(dev) for t in lg_h]
    xb = [t.to(dev) for t in x_h]
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    plans = [M.RoutePlan.allocate(T, E, k, device=dev) for _ in range(G)]
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_PREFILL, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    ev = [(_graph_event(), _graph_event(), _graph_event()) for _ in range(G)]
    residual = args.output == "residual"

    def step(g):
        e0, e1, e2 = ev[g]
        flush.fill_(g)  # larger than L2: every step starts from a cold L2
        e0.record(stream)
        M.moe_route_plan(lg[g], k, plans[g], stream=stream, with_counts_host=False)
        e1.record(stream)
        M.moe_expert_ffn(pool, 0, xb[g], plans[g], slot_of, out, ws, path=M.MOE_PATH_PREFILL, stream=stream,
                         accumulate=residual)
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
    soak_n = 0
    if soak_s > 0:
        soak_n, _ = _soak(lambda n: graphs[n % G].replay(), soak_s)
    total = 0.0
    for i in range(args.steps):
        graphs[i % G].replay()
        torch.cuda.synchronize()
        e0, e1, e2 = ev[i % G]
        route_ms.append(e0.elapsed_time(e1))
        ffn_ms.append(e1.elapsed_time(e2))
        total += e0.elapsed_time(e2)
    clk = clocks.stop()
    res = dict(step_ms=total / args.steps, route_ms=route_ms, ffn_ms=ffn_ms, clocks=clk, soak_steps=soak_n)

    # end to end through the C ABI
    lg_pin = [t.pin_memory() for t in lg_h]
    x_pin = [t.pin_memory() for t in x_h]
    out_pin = [torch.empty((T, H), dtype=torch.float32).pin_memory() for _ in range(2)]
    lg_dev = [torch.empty((T, E), dtype=torch.float32, device=dev) for _ in range(2)]
    x_dev = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    out_dev = [torch.empty((T, H), dtype=torch.float32, device=dev) for _ in range(2)]
    compute = torch.cuda.Stream(device=dev)
    copy = torch.cuda.Stream(device=dev)
    up_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]
    n_steps = args.warmup + args.steps

    def upload(g):
        b = g % 2
        with torch.cuda.stream(copy):
            copy.wait_event(comp_done[b]) if g >= 2 else None
            lg_dev[b].copy_(lg_pin[g % G], non_blocking=True)
            x_dev[b].copy_(x_pin[g % G], non_blocking=True)
            up_done[b].record(copy)

    def run(g):
        b = g % 2
        compute.wait_event(up_done[b])
        if g >= 2:
            compute.wait_event(down_done[b])  # out_dev[b] read back
        M.moe_route_plan(lg_dev[b], k, plans[b], stream=compute, with_counts_host=False)
        M.moe_expert_ffn(pool, 0, x_dev[b], plans[b], slot_of, out_dev[b], ws, path=M.MOE_PATH_PREFILL,
                         stream=compute)
        comp_done[b].record(compute)
        with torch.cuda.stream(copy):
            copy.wait_event(comp_done[b])
            out_pin[b].copy_(out_dev[b], non_blocking=True)
            down_done[b].record(copy)

    def e2e_run(n):
        upload(0)
        for g in range(n):
            if g + 1 < n:
                upload(g + 1)
            run(g)
        torch.cuda.synchronize()

    e2e_run(args.warmup)
    t0 = time.perf_counter()
    e2e_run(args.steps)
    e2e_ms = (time.perf_counter() - t0) / args.steps * 1e3
    res.update(e2e_ms=e2e_ms, h2d=lg_pin[0].numel() * 4 + x_pin[0].numel() * 2, d2h=out_pin[0].numel() * 4)
    pool.close()
    del slots, flush
    torch.cuda.empty_cache()
    return res


def gguf_obj(args, fmt, wid=4, layers=24):
    """Decode on GGUF expert weights read in place: Qwen-30B-A3B-shaped
    layers (128 experts, top-8) resident in GGUF form, one token per step
    through ``layers`` layers back to back (each layer its own copy of the
    experts at its own addresses and its own logits and activations, so a
    layer's rows were last read ``layers`` - 1 layers earlier: about 0.5 GB
    in between, well over L2).  The timed step is ``layers`` calls of
    moe_decode_layer_gguf (routing and the experts in one launch each),
    graph-captured; moe_route_plan + moe_expert_ffn_gguf (two calls per
    layer) is timed beside it.  HBM bytes per layer: the routed experts'
    GGUF rows (gate, up, down)."""
    import torch

    import oracle
    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[wid]
    dev = torch.device("cuda", torch.cuda.current_device())
    E, k, H, I, L = wl.experts, wl.top_k, wl.hidden, wl.inter, layers
    eb = M.moe_gguf_expert_bytes(fmt, H, I)
    img = torch.empty(E * eb, dtype=torch.uint8).pin_memory()
    for e in range(E):
        M.pack_gguf_expert(S.expert_weights_gguf(wl, fmt, 0, e), fmt, H, I, img.data_ptr() + e * eb)
    slots = torch.empty((L, E * eb), dtype=torch.uint8, device=dev)
    slots[0].copy_(img)
    for l in range(1, L):
        slots[l].copy_(slots[0])
    slot_of = torch.arange(E, dtype=torch.int32, device=dev)
    G = args.warmup + args.steps
    lg = torch.from_numpy(S.logits(wl, 0, 0, G * L).reshape(G, L, 1, E)).to(dev)
    xb = torch.from_numpy(S.activations_bf16_bits(wl, 0, 0, G * L).view(np.int16).reshape(G, L, 1, H)).to(dev)
    xb = xb.view(torch.bfloat16)
    out = torch.zeros((1, H), dtype=torch.float32, device=dev)
    plan = M.RoutePlan.allocate(1, E, k, device=dev)
    ws = M.alloc_gguf_workspace(1, k, H, I, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def timed(call):
        ev = [(_graph_event(), _graph_event()) for _ in range(G)]

        def step(g):
            ev[g][0].record(stream)
            for l in range(L):
                call(g, l)
            ev[g][1].record(stream)

        with torch.cuda.stream(stream):
            step(0)
        stream.synchronize()
        graphs = []
        for g in range(G):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                step(g)
            graphs.append(gr)
        for g in range(args.warmup):
            graphs[g].replay()
        torch.cuda.synchronize()
        times = []
        for g in range(args.warmup, G):
            graphs[g].replay()
            torch.cuda.synchronize()
            times.append(ev[g][0].elapsed_time(ev[g][1]))
        return statistics.median(times)

    def fused(g, l):
        M.moe_decode_layer_gguf(fmt, slots[l], E, H, I, lg[g, l], xb[g, l], plan, slot_of, E, out, ws,
                                accumulate=True, stream=stream)

    def two_calls(g, l):
        M.moe_route_plan(lg[g, l], k, plan, stream=stream, with_counts_host=False)
        M.moe_expert_ffn_gguf(fmt, slots[l], E, H, I, xb[g, l], plan, slot_of, E, out, ws, accumulate=True,
                              stream=stream)

    ms = timed(fused)
    ms_two = timed(two_calls)
    status = M.moe_ffn_status(ws, M.MOE_PATH_DECODE, stream=stream)
    if status:
        raise RuntimeError(f"GGUF decode: status bits {status:#x}")
    rbh, rbi = oracle.gguf_row_bytes(fmt, H), oracle.gguf_row_bytes(fmt, I)
    layer_bytes = k * (2 * I * rbh + H * rbi)
    hbm_peak, _, peak_kind = _peaks()
    achieved = layer_bytes / (ms / L / 1e3) / 1e9
    del slots
    torch.cuda.empty_cache()
    return {"workload": f"{wl.name}_decode_gguf_{fmt}", "value": 1e3 / ms, "unit": f"tokens/s ({L} layers)",
            "ms_per_step": ms, "us_per_layer": ms / L * 1e3,
            "config": {"hidden": H, "inter": I, "experts": E, "top_k": k, "tokens_per_step": 1, "format": fmt,
                       "layers": L, "l2": f"{L} layers, each its own copy of the experts (no layer's rows in L2)",
                       "timing": f"{L} x moe_decode_layer_gguf (one launch each), graph per step, CUDA events"},
            "route_plus_ffn_us_per_layer": ms_two / L * 1e3,
            "roofline": {"kernel": "gguf_fused_kernel: one launch per layer (routing, gate/up+SwiGLU, down, combine)",
                         "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "peak_kind": peak_kind,
                         "traffic": NCU_TRAFFIC.get(f"gguf_fused_kernel/{fmt}") if wid == 4 else None,
                         "algorithmic_bytes_per_launch": layer_bytes},
            "gpu_launches": args.steps * L}


def tiny_obj(args, threads):
    """Config 0 (hidden 256, inter 512, 8 experts, top-2, 16 tokens, all
    resident): the layer on both GPU paths (routing + expert FFN, graph,
    CUDA events) and the oracle on one thread and on every host core."""
    import torch

    import oracle
    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[0]
    dev = torch.device("cuda", torch.cuda.current_device())
    E, k, H, I, T = wl.experts, wl.top_k, wl.hidden, wl.inter, wl.tokens
    host, slots, pool = _prefill_setup(M, wl, dev)
    slot_of = torch.arange(E, dtype=torch.int32, device=dev)
    lg = torch.from_numpy(S.logits(wl, 0)).to(dev)
    x = torch.from_numpy(S.activations_bf16_bits(wl, 0).view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    plan = M.RoutePlan.allocate(T, E, k, device=dev)
    res = {"workload": wl.name, "config": {"hidden": H, "inter": I, "experts": E, "top_k": k, "tokens": T}}
    stream = torch.cuda.Stream(device=dev)
    for name, path in (("decode_path", M.MOE_PATH_DECODE), ("prefill_path", M.MOE_PATH_PREFILL)):
        ws = M.alloc_ffn_workspace(T, k, H, I, path, device=dev)

        def step():
            M.moe_route_plan(lg, k, plan, stream=stream, with_counts_host=False)
            M.moe_expert_ffn(pool, 0, x, plan, slot_of, out, ws, path=path, stream=stream)

        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step()
        for _ in range(args.warmup):
            gr.replay()
        torch.cuda.synchronize()
        a, b = _events()
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(args.steps):
                gr.replay()
            b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) / args.steps * 1e3
        res[name] = {"us_per_layer_call": us, "tokens_per_s": T / (us / 1e6)}
    # the decode step as one launch: routing inside the kernel (moe_decode_layer)
    ws = M.alloc_ffn_workspace(T, k, H, I, M.MOE_PATH_DECODE, device=dev)

    def fused_step():
        M.moe_decode_layer(pool, 0, lg, x, plan, slot_of, out, ws, stream=stream)

    with torch.cuda.stream(stream):
        fused_step()
    stream.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        fused_step()
    for _ in range(args.warmup):
        gr.replay()
    torch.cuda.synchronize()
    a, b = _events()
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(args.steps):
            gr.replay()
        b.record(stream)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / args.steps * 1e3
    res["decode_layer"] = {"us_per_layer_call": us, "tokens_per_s": T / (us / 1e6),
                           "how": "moe_decode_layer: routing and the experts in one launch"}
    ws_all = S.stack_experts(S.layer_weights(wl, 0))
    lgh, xbh = S.logits(wl, 0), S.activations_bf16_bits(wl, 0)
    cpu = {}
    for n in (1, threads):
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 1.0:
            ids, w = oracle.route(lgh, k)
            oracle.hist_perm(ids, E)
            oracle.layer(xbh, ids, w, ws_all, prefill=False, threads=n)
            reps += 1
        cpu[n] = reps * T / (time.perf_counter() - t0)
    res["cpu_baseline"] = {"value": cpu[threads], "unit": "tokens/s", "cores": threads, "kind": "oracle",
                           "sample": "the whole layer (16 tokens, decode-path arithmetic), repeated for a second",
                           "single_thread_value": cpu[1]}
    pool.close()
    return res


def prefill_obj(args, wl, mma, threads, cpu=True):
    res = prefill_timing(args, wl, soak_s=args.soak / 2)
    flops = 6.0 * wl.hidden * wl.inter * wl.tokens * wl.top_k
    ffn_s = statistics.median(res["ffn_ms"]) / 1e3
    achieved = flops / ffn_s / 1e12
    _, bf16_peak, peak_kind = _peaks()
    fp4_peak = bf16_peak * FP4_OVER_BF16
    obj = {"workload": wl.name, "value": wl.tokens / (res["step_ms"] / 1e3), "unit": "tokens/s",
           "ms_per_step": res["step_ms"], "dtype": "mxf8f6f4->f32",
           "config": {"hidden": wl.hidden, "inter": wl.inter, "experts": wl.experts, "top_k": wl.top_k,
                      "tokens": wl.tokens, "l2": "256 MB flush before every step",
                      "output": ("added into a residual stream (MOE_FFN_ACCUMULATE)" if args.output == "residual"
                                 else "overwritten (out zeroed, then the combine adds into it)")},
           "roofline": {"kernel": "prefill expert FFN (MXFP8 quant, gate/up GEMM, down GEMM with the combine in "
                                  "its epilogue)",
                        "bound": "tensor", "achieved": achieved, "peak": mma["burst_tflops"], "unit": "TFLOP/s",
                        "frac": achieved / mma["burst_tflops"],
                        "peak_kind": "measured rate of tcgen05.mma kind::mxf8f6f4 on this GPU (peaks.mxf8f6f4)",
                        "frac_of_mxfp4_peak": achieved / fp4_peak,
                        "mxfp4_peak": fp4_peak,
                        "mxfp4_peak_kind": f"{peak_kind} bf16 x {FP4_OVER_BF16:g} (published dense ratio); the "
                                           "kind::mxf4 MMA is not built, so it is not measured",
                        "traffic": NCU_TRAFFIC.get("grouped_gemm_tc_kernel/" + wl.name),
                        "traffic_scope": "DRAM bytes of the two GEMM launches of one layer",
                        "algorithmic_flops_per_launch": flops, "avg_launch_us": ffn_s * 1e6},
           "kernels_us": {"route_plan": statistics.median(res["route_ms"]) * 1e3, "expert_ffn": ffn_s * 1e6},
           "ffn_times": {"median_ms": statistics.median(res["ffn_ms"]),
                         "cv": (statistics.pstdev(res["ffn_ms"]) / statistics.mean(res["ffn_ms"])
                                if len(res["ffn_ms"]) > 1 else 0.0)},
           "e2e": {"value": wl.tokens / (res["e2e_ms"] / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": res["h2d"],
                   "d2h_bytes_per_step": res["d2h"],
                   "how": "moe_route_plan + moe_expert_ffn through the C ABI; logits and x from pinned host memory, "
                          "out back to pinned host memory, uploads and read-backs on a second stream overlapping "
                          "the neighbouring steps' compute; host clock over the steps"},
           # per step: routing (top-k and scatter passes), quantisation, two GEMMs
           "gpu_launches": args.steps * 5,
           "clocks": res["clocks"]}
    if cpu:
        obj["cpu_baseline"] = cpu_prefill_baseline(wl, args.cpu_prefill_tokens.get(wl.wid, 32), threads)
    return obj


def staged_prefill_leg(args, wl):
    """Prefill of one layer through a pool of ``--prefill-slots`` slots (fewer
    than the routed experts), every expert in pinned host memory: per step,
    routing on the GPU, then moe_prefill_staged (windows of unique experts
    staged on a copy stream while the previous window's grouped GEMMs run).
    Timed end to end on the host clock and by CUDA events on the compute
    stream: x and logits come from pinned host memory, out goes back there."""
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
        a, b = _events()
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


def _standalone_line(obj, args):
    """One workload's sub-object as a line of its own (``--workload N``)."""
    line = {"metric": METRIC, "value": obj["value"], "unit": obj["unit"], "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": obj["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": obj.get("dtype", "f32"), "data": "synthetic",
            "config": dict(workload=obj["workload"], **obj["config"])}
    for key in ("roofline", "kernels_us", "ffn_times", "staging", "host_planned", "same_events_as_host_planned",
                "outputs_vs_host_planned_rel_l2", "e2e", "gpu_launches", "clocks", "cpu_baseline"):
        if key in obj:
            line[key] = obj[key]
    return line


def reference_arm(args, wl, threads, rank):
    """The CPU oracle as it stands, on the host cores: every step is one
    decode token through a sample of ``--cpu-layers`` of the 24 layers (the
    same layers each step, distinct tokens), timed on the host clock; the
    value is tokens/s of that sample (a step is that fraction of a token)."""
    if rank != 0:
        return
    import oracle

    oracle.build()
    layers = _sample_layers(wl, args.cpu_layers)
    cache = {l: S.stack_experts(S.layer_weights(wl, l)) for l in layers}
    times = [_oracle_decode_sample(wl, s % wl.steps, layers, cache, threads)
             for s in range(args.warmup + args.steps)]
    timed = times[args.warmup:]
    ms_step = statistics.mean(timed) * 1e3
    frac = len(layers) / wl.layers
    v = frac / (ms_step / 1e3)
    sample = (f"each step: 1 decode token through {len(layers)} of {wl.layers} layers (layers {layers}), i.e. "
              f"{frac:.4g} of a token; value = that fraction over the step time")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": _decode_config(wl, args, 1),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def _decode_config(wl, args, world):
    return {"workload": wl.name, "layers": wl.layers, "hidden": wl.hidden, "inter": wl.inter,
            "experts": wl.experts, "top_k": wl.top_k, "tokens_per_step": 1,
            "resident_experts": wl.layers * wl.experts,
            "l2": "inputs larger than L2: each step reads 96 distinct experts (1.27 GB) of a 10.2 GB set",
            "output": ("each layer adds into the step's residual row (moe_decode_layer_acc)"
                       if args.output == "residual" else "each layer overwrites its own output (moe_decode_layer)"),
            "parallelism": f"replicas{world}"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-layers", type=int, default=4, help="layers per oracle decode sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="default run: skip the prefill, offload and peak parts")
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of back-to-back steps around each timed region while clocks are sampled")
    ap.add_argument("--workload", type=int, default=1, choices=[1, 2, 3, 4],
                    help="1: the default line (decode headline + prefill/offload parts); 2, 3, 4: one line for "
                         "that workload alone")
    ap.add_argument("--policy", default="lru", choices=["lru", "fifo", "lfu", "lfru", "slru"],
                    help="eviction policy of the offload pool (workload 2)")
    ap.add_argument("--stage-parts", default="decode", choices=["whole", "decode"],
                    help="workload 2: copy only what the decode kernel reads (MOE_STAGE_DECODE: the gate/up rows "
                         "and the column-blocked down copy), or whole packed experts")
    ap.add_argument("--output", default="residual", choices=["residual", "overwrite"],
                    help="decode: each layer adds into the step's residual row (moe_decode_layer_acc) or "
                         "overwrites its own output (moe_decode_layer); prefill: out += or out =")
    ap.add_argument("--prefetch", type=int, default=0,
                    help="workload 2: after each layer's staging, prefetch up to this many experts of the next layer")
    ap.add_argument("--prefill-slots", type=int, default=None,
                    help="workloads 3/4: run the layer through a pool of this many slots (moe_prefill_staged)")
    ap.add_argument("--window", type=int, default=None,
                    help="with --prefill-slots: unique experts per staging window (default slots // 2)")
    ap.add_argument("--policy-sweep", action="store_true",
                    help="with --workload 2: also replay the whole routing stream under every policy")
    ap.add_argument("--gguf-only", action="store_true",
                    help="run only the GGUF decode legs (both formats) and print their JSON line")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers (smaller case for profiler captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    # oracle samples of the prefill workloads: tokens of the layer (about
    # 10 s of CPU work each on 16 cores)
    args.cpu_prefill_tokens = {3: 48, 4: 96}
    world, rank, local = _dist()
    threads = os.cpu_count() or 1
    wl = S.WORKLOADS[args.workload]
    if args.impl == "reference":
        reference_arm(args, S.WORKLOADS[1], threads, rank)
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
    import routed_expert_ffn_histogram_gb300 as M

    if args.gguf_only:
        if rank == 0:
            print(json.dumps({"gguf_decode": {fmt: gguf_obj(args, fmt) for fmt in ("q4_k", "q8_0")}}))
        return

    dev = torch.device("cuda", torch.cuda.current_device())
    if args.workload == 2:
        host = build_host_store(M, wl, wl.layers if args.layers is None else min(args.layers, wl.layers))
        obj = offload_obj(args, wl, host)
        line = _standalone_line(obj, args)
        if args.policy_sweep:
            line["policy_sweep"] = policy_sweep(wl, obj["config"]["layers"], dev)
        print(json.dumps(line))
        return
    if args.workload in (3, 4):
        if args.prefill_slots:
            staged_prefill_leg(args, wl)
            return
        mma = measure_mma_peak(dev)
        obj = prefill_obj(args, wl, mma, threads, cpu=not args.no_cpu_baseline)
        line = _standalone_line(obj, args)
        line["peaks"] = {"mxf8f6f4": mma}
        print(json.dumps(line))
        return

    # ---- the default line: decode headline, then the other parts ----
    if args.layers:
        import dataclasses

        wl = dataclasses.replace(wl, layers=min(args.layers, wl.layers))
    hbm_peak, _, peak_kind = _peaks()
    host = build_host_store(M, wl, wl.layers)
    res = gpu_decode_leg(args, wl, host, rank, world)
    ms = res["elapsed_ms"] / args.steps
    e2e_ms = res["e2e_ms"] / args.steps
    ms, e2e_ms = reduce_max_over_ranks([ms, e2e_ms], world, device="cuda")
    layer_bytes = wl.top_k * 3 * (wl.hidden * wl.inter // 2 + wl.hidden * wl.inter // 32)
    # per-launch duration: the timed steps are back-to-back launches of the
    # decode kernel on this stream (one CUDA graph per step), so step time /
    # launches per step
    launch_s = ms / 1e3 / wl.layers
    achieved = layer_bytes / launch_s / 1e9
    line = {"metric": METRIC, "value": world * 1e3 / ms, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": _decode_config(wl, args, world),
            "formats": "weights MXFP4 (E2M1 + E8M0 per 32), activations bf16, fp32 accumulation",
            "roofline": {"kernel": "decode_fused_kernel: one launch per layer (routing, gate/up+SwiGLU, "
                                   "down+combine)",
                         "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "peak_kind": peak_kind,
                         "traffic": NCU_TRAFFIC["decode_fused_kernel"],
                         "algorithmic_bytes_per_launch": layer_bytes,
                         "avg_launch_us": launch_s * 1e6},
            "kernels_us": {"decode_layer": launch_s * 1e6},
            "step_times": {"median_ms": statistics.median(res["step_ms"]),
                           "cv": (statistics.pstdev(res["step_ms"]) / statistics.mean(res["step_ms"])
                                  if len(res["step_ms"]) > 1 else 0.0),
                           "how": "the K steps again, each between its own pair of CUDA events"},
            "e2e": {"value": world * 1e3 / e2e_ms, "unit": "tokens/s", "h2d_bytes_per_step": res["h2d"],
                    "d2h_bytes_per_step": res["d2h"], "matches_graph_outputs": res["e2e_matches_graph"],
                    "how": "moe_decode_layer_acc x 24 per step through the C ABI (one captured graph per staging "
                           "buffer set); each step's logits, activations and residual row uploaded from pinned "
                           "memory and its row read back to pinned memory, on a copy stream overlapping the "
                           "neighbouring steps' compute; host clock until the last row is in host memory"},
            "gpu_launches": args.steps * wl.layers,
            "clocks": dict(res["clocks"] or {}, window="sampled over a soak of the same step graphs "
                                                       f"({res['soak']['steps']} steps, "
                                                       f"{res['soak']['seconds']:.2f} s) enclosing the timed region")
            if res["clocks"] else None}
    if not args.no_cpu_baseline and rank == 0:
        import oracle

        oracle.build()
        line["cpu_baseline"] = cpu_decode_baseline(wl, args.cpu_layers, threads, steps=2)
    if world == 1 and not args.decode_only and args.layers is None:
        mma = measure_mma_peak(dev)
        link_peak = _pinned_link_peak(dev)
        line["peaks"] = {"mxf8f6f4": mma, "pinned_h2d_gbs": link_peak,
                         "hbm_gbs": hbm_peak, "hbm_kind": peak_kind,
                         "mxfp4_tflops": _peaks()[1] * FP4_OVER_BF16,
                         "mxfp4_kind": "measured bf16 x 6 (published dense ratio; kind::mxf4 not built)"}
        line["prefill"] = {}
        for wid in (3, 4):
            pw = S.WORKLOADS[wid]
            line["prefill"][pw.name] = prefill_obj(args, pw, mma, threads, cpu=not args.no_cpu_baseline)
        ow = S.WORKLOADS[2]
        off = offload_obj(args, ow, host)
        if not args.no_cpu_baseline:
            off["cpu_baseline"] = cpu_offload_baseline(ow, args.cpu_layers, threads)
        line["offload"] = {ow.name: off}
        line["gguf_decode"] = {fmt: gguf_obj(args, fmt) for fmt in ("q4_k", "q8_0")}
        line["tiny"] = tiny_obj(args, threads)
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
