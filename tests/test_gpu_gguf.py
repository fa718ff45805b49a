"""GPU parity of the decode layer on GGUF expert weights (Q8_0, Q4_K) read
in place (moe_expert_ffn_gguf, moe_decode_layer_gguf) against the oracle's
GGUF layer (oracle.layer_gguf, reading r22): the SwiGLU output h within one
bf16 ulp and the layer output within the decode path's rel-L2 bound, at the
Qwen-30B-A3B shape (both formats, the single-launch kernel), the GPT-OSS
shape (Q8_0: rows of 3060 bytes take the three-launch path) and the tiny
shape (single launch up to 32 assignments, three launches beyond);
accumulate mode, a routed expert without a slot, fused routing equal to
moe_route_plan, bitwise-repeatable output, counters left zero, and the
shape refusals."""
import numpy as np
import pytest

import moe_synth as S
import oracle
from helpers import rel_l2
from test_gpu_decode import DECODE_REL_L2

pytestmark = pytest.mark.gpu


def _bf16_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_h(h, href):
    """h is bf16(silu(g) u) of fp32 sums g, u: only the fp32 summation order
    differs from the oracle, which moves a rounding of bf16(h) now and then
    -- by one ulp, or by a few ulps of a value near zero that g * u nearly
    cancels to.  So: more than 99 % bit-exact, and every value within one
    ulp of the oracle's or within 2^-12 of the rms of h."""
    a, b = _bf16_f64(h), _bf16_f64(href)
    assert (np.asarray(h) == np.asarray(href)).mean() > 0.99
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(b), 1e-38))) - 7)
    tol = np.maximum(ulp, np.sqrt(np.mean(b * b)) * 2.0 ** -12)
    assert np.all(np.abs(a - b) <= tol)


def _setup(M, wl, fmt, T, layer=0, step=0):
    """GGUF slots holding the routed experts of T tokens; returns what the
    GPU call and the oracle need."""
    import torch

    E, k, H, I = wl.experts, wl.top_k, wl.hidden, wl.inter
    logits = S.logits(wl, layer, step, T)
    xb = S.activations_bf16_bits(wl, layer, step, T)
    ids, w = oracle.route(logits, k)
    used = sorted(set(ids.reshape(-1).tolist()))
    eb = M.moe_gguf_expert_bytes(fmt, H, I)
    img = np.zeros(len(used) * eb, np.uint8)
    rbh, rbi = oracle.gguf_row_bytes(fmt, H), oracle.gguf_row_bytes(fmt, I)
    stacked = dict(gate=np.zeros((E, I, rbh), np.uint8), up=np.zeros((E, I, rbh), np.uint8),
                   down=np.zeros((E, H, rbi), np.uint8))
    slot_of = np.full(E, -1, np.int32)
    for s, e in enumerate(used):
        wt = S.expert_weights_gguf(wl, fmt, layer, e)
        M.pack_gguf_expert(wt, fmt, H, I, img[s * eb:(s + 1) * eb])
        for key in stacked:
            stacked[key][e] = wt[key]
        slot_of[e] = s
    slots = torch.from_numpy(img).cuda()
    lg = torch.from_numpy(logits).cuda()
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    plan = M.RoutePlan.allocate(T, E, k)
    M.moe_route_plan(lg, k, plan)
    return dict(slots=slots, n_slots=len(used), x=x, plan=plan, slot_of=torch.from_numpy(slot_of).cuda(),
                xb=xb, ids=ids, w=w, stacked=stacked, used=used)


def _run(M, wl, fmt, c, accumulate=False, out=None):
    import torch

    T = c["x"].shape[0]
    ws = M.alloc_gguf_workspace(T, wl.top_k, wl.hidden, wl.inter)
    if out is None:
        out = torch.empty((T, wl.hidden), dtype=torch.float32, device="cuda")
    M.moe_expert_ffn_gguf(fmt, c["slots"], c["n_slots"], wl.hidden, wl.inter, c["x"], c["plan"], c["slot_of"],
                          wl.experts, out, ws, accumulate=accumulate)
    torch.cuda.synchronize()
    h = M.gguf_workspace_h(ws, T, wl.top_k, wl.inter).cpu().numpy().view(np.uint16)
    assert M.moe_ffn_status(ws, M.MOE_PATH_DECODE) == 0
    return out.cpu().numpy(), h


@pytest.mark.parametrize("fmt,wid,T", [("q4_k", 4, 1), ("q8_0", 4, 1), ("q4_k", 4, 3), ("q8_0", 4, 4),
                                       ("q8_0", 1, 1), ("q8_0", 0, 16), ("q4_k", 0, 16), ("q4_k", 0, 17),
                                       ("q8_0", 0, 20)])
def test_gguf_layer_matches_oracle(fmt, wid, T):
    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[wid]
    c = _setup(M, wl, fmt, T)
    assert np.array_equal(c["plan"].ids.cpu().numpy(), c["ids"])
    got, h = _run(M, wl, fmt, c)
    ref, href = oracle.layer_gguf(fmt, c["xb"], c["ids"], c["w"], c["stacked"], threads=16, want_h=True)
    _check_h(h, href)
    assert rel_l2(got, ref) <= DECODE_REL_L2


def test_gguf_accumulate_and_missing_slot():
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl, fmt, T = S.WORKLOADS[0], "q4_k", 4
    c = _setup(M, wl, fmt, T)
    ref = oracle.layer_gguf(fmt, c["xb"], c["ids"], c["w"], c["stacked"], threads=16)
    base = torch.full((T, wl.hidden), 0.5, dtype=torch.float32, device="cuda")
    got, _ = _run(M, wl, fmt, c, accumulate=True, out=base)
    assert rel_l2(got - 0.5, ref) <= DECODE_REL_L2
    # an expert routed for token 0 loses its slot: token 0 becomes NaN,
    # tokens that do not route to it stay finite
    e0 = int(c["ids"][0, 0])
    c["slot_of"][e0] = -1
    got, _ = _run(M, wl, fmt, c)
    assert np.isnan(got[0]).all()
    clean = [t for t in range(T) if e0 not in c["ids"][t].tolist()]
    assert clean and np.isfinite(got[clean]).all()


def test_gguf_shape_refusals():
    import ctypes

    import routed_expert_ffn_histogram_gb300 as M

    L = M.lib()
    n = ctypes.c_size_t(0)
    # Q4_K blocks are 256 long: the GPT-OSS hidden size 2880 does not fit
    assert L.moe_gguf_expert_bytes(M.MOE_GGUF_Q4_K, 2880, 2880, ctypes.byref(n)) == M.MOE_ERR_INVALID
    assert L.moe_gguf_expert_bytes(7, 2048, 768, ctypes.byref(n)) == M.MOE_ERR_INVALID
    assert L.moe_gguf_expert_bytes(M.MOE_GGUF_Q8_0, 2880, 2880, ctypes.byref(n)) == M.MOE_OK
    assert n.value == 256 * ((2 * 2880 * 90 * 34 + 2880 * 90 * 34 + 255) // 256)
    assert L.moe_expert_ffn_gguf(M.MOE_GGUF_Q4_K, 256, 1, 2880, 2880, 256, 1, 4, 1, 1, 1, 32, 256, 1 << 20, 256,
                                 0, None) == M.MOE_ERR_INVALID


def _counters_zero(M, ws, T, k, H, I):
    """The control block of a GGUF workspace (ticket, status, per-assignment
    counters of h rows) is all zero."""
    import torch

    return not ws[:256].view(torch.int32).cpu().numpy().any()


@pytest.mark.parametrize("fmt,wid,T", [("q4_k", 4, 1), ("q8_0", 4, 1), ("q4_k", 4, 4), ("q8_0", 0, 16)])
def test_gguf_decode_layer_fused_routing(fmt, wid, T):
    """moe_decode_layer_gguf: routing outputs equal moe_route_plan's bit for
    bit, the layer equals the oracle's, repeated calls give the same bits
    (no floating-point atomics), and the counters are zero afterwards."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[wid]
    E, k, H, I = wl.experts, wl.top_k, wl.hidden, wl.inter
    c = _setup(M, wl, fmt, T)
    lg = torch.from_numpy(S.logits(wl, 0, 0, T)).cuda()
    plan = M.RoutePlan.allocate(T, E, k)
    ws = M.alloc_gguf_workspace(T, k, H, I)
    outs = []
    for _ in range(3):
        out = torch.full((T, H), 7.0, dtype=torch.float32, device="cuda")
        M.moe_decode_layer_gguf(fmt, c["slots"], c["n_slots"], H, I, lg, c["x"], plan, c["slot_of"], E, out, ws)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
        assert _counters_zero(M, ws, T, k, H, I)
    for name in ("ids", "w", "counts", "offsets", "perm", "inv"):
        assert np.array_equal(getattr(plan, name).cpu().numpy(), getattr(c["plan"], name).cpu().numpy()), name
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    ref, href = oracle.layer_gguf(fmt, c["xb"], c["ids"], c["w"], c["stacked"], threads=16, want_h=True)
    _check_h(M.gguf_workspace_h(ws, T, k, I).cpu().numpy().view(np.uint16), href)
    assert rel_l2(outs[0], ref) <= DECODE_REL_L2
    assert M.moe_ffn_status(ws, M.MOE_PATH_DECODE) == 0
    # accumulate: out += layer
    base = torch.full((T, H), 0.25, dtype=torch.float32, device="cuda")
    M.moe_decode_layer_gguf(fmt, c["slots"], c["n_slots"], H, I, lg, c["x"], plan, c["slot_of"], E, base, ws,
                            accumulate=True)
    assert rel_l2(base.cpu().numpy() - 0.25, ref) <= DECODE_REL_L2


def test_gguf_decode_layer_many_experts_and_tokens():
    """The fused GGUF kernel's routing with 256 experts (eight candidates a
    lane) and several routing warps (4 tokens): routing outputs equal
    moe_route_plan's bit for bit and the layer equals the oracle's."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    base = S.WORKLOADS[0]
    wl = S.Workload(0, "gguf_e256", 1, base.hidden, base.inter, 256, 4, 4, 1, 256, 0.0, 0)
    fmt, T, E, k, H, I = "q8_0", 4, 256, 4, base.hidden, base.inter
    c = _setup(M, wl, fmt, T)
    lg = torch.from_numpy(S.logits(wl, 0, 0, T)).cuda()
    plan = M.RoutePlan.allocate(T, E, k)
    ws = M.alloc_gguf_workspace(T, k, H, I)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    M.moe_decode_layer_gguf(fmt, c["slots"], c["n_slots"], H, I, lg, c["x"], plan, c["slot_of"], E, out, ws)
    torch.cuda.synchronize()
    for name in ("ids", "w", "counts", "offsets", "perm", "inv"):
        assert np.array_equal(getattr(plan, name).cpu().numpy(), getattr(c["plan"], name).cpu().numpy()), name
    ref = oracle.layer_gguf(fmt, c["xb"], c["ids"], c["w"], c["stacked"], threads=16)
    assert rel_l2(out.cpu().numpy(), ref) <= DECODE_REL_L2
    assert _counters_zero(M, ws, T, k, H, I)


def test_gguf_single_launch_matches_three_launch():
    """The same layer through the single-launch kernel (8 tokens x top-2 =
    16 assignments) and the three-launch path (24 tokens: 48 assignments):
    the first 8 tokens' outputs agree to fp32 summation order."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl, fmt = S.WORKLOADS[0], "q4_k"
    c = _setup(M, wl, fmt, 24)
    big, _ = _run(M, wl, fmt, c)
    small_plan = M.RoutePlan.allocate(8, wl.experts, wl.top_k)
    M.moe_route_plan(torch.from_numpy(S.logits(wl, 0, 0, 24)[:8]).cuda(), wl.top_k, small_plan)
    ws = M.alloc_gguf_workspace(8, wl.top_k, wl.hidden, wl.inter)
    out = torch.empty((8, wl.hidden), dtype=torch.float32, device="cuda")
    M.moe_expert_ffn_gguf(fmt, c["slots"], c["n_slots"], wl.hidden, wl.inter, c["x"][:8], small_plan, c["slot_of"],
                          wl.experts, out, ws)
    assert rel_l2(out.cpu().numpy(), big[:8]) <= 1e-5
