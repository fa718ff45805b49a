"""Pins of the oracle's expert FFN, MXFP4 GEMV, SwiGLU and combine: an
integer-exact special case (bit-exact against integer matmul), float64 numpy
evaluations within the fp32 summation bound, torch's float64 silu, and torch
casts for the bf16 / E4M3 rounding steps."""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def _pack(int_codes):
    """[rows][K] nibble codes -> canonical bytes (even element in the low nibble)."""
    c = int_codes.astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _deq64(codes, scales):
    lo, hi = codes & 15, codes >> 4
    el = np.empty((codes.shape[0], codes.shape[1] * 2))
    el[:, 0::2] = E2M1[lo]
    el[:, 1::2] = E2M1[hi]
    return el * np.exp2(np.repeat(scales.astype(np.float64) - 127, 32, axis=1))


def _bf16_bits(f):
    return torch.from_numpy(np.asarray(f, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_f32(b):
    return torch.from_numpy(np.asarray(b, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


def _int_expert(rng, H, I):
    """Weights whose elements are in {0, +-1, +-2} x {1/2, 1, 2}: every sum of
    products with small-integer activations is exact in fp32."""
    pick = np.array([0, 2, 4, 10, 12])                      # 0, 1, 2, -1, -2
    val = {0: 0, 2: 1, 4: 2, 10: -1, 12: -2}
    out = {}
    for name, rows, K in [("gate", I, H), ("up", I, H), ("down", H, I)]:
        nib = pick[rng.integers(0, 5, (rows, K))]
        sc = (126 + rng.integers(0, 3, (rows, K // 32))).astype(np.uint8)
        out[name + "_codes"] = _pack(nib)
        out[name + "_scales"] = sc
        ints = np.vectorize(val.get)(nib).astype(np.int64)
        out[name + "_x4"] = ints * (np.repeat(2 ** (sc.astype(np.int64) - 126), 32, axis=1))  # 2*W
    return out


def test_gemv_integer_exact():
    rng = np.random.default_rng(11)
    H, I = 96, 64
    wt = _int_expert(rng, H, I)
    x = rng.integers(-3, 4, H).astype(np.float32)
    g, u, _ = oracle.expert_gateup(wt, x)
    g_ref = (wt["gate_x4"] @ x.astype(np.int64)) / 2
    u_ref = (wt["up_x4"] @ x.astype(np.int64)) / 2
    assert np.array_equal(g.astype(np.float64), g_ref)
    assert np.array_equal(u.astype(np.float64), u_ref)
    h = rng.integers(-5, 6, I).astype(np.float32)
    y = oracle.expert_down(wt, h)
    assert np.array_equal(y.astype(np.float64), (wt["down_x4"] @ h.astype(np.int64)) / 2)


def test_gateup_float64_bound_and_swiglu():
    wl = S.WORKLOADS[0]
    wt = S.expert_weights(wl, 0, 3)
    xb = S.activations_bf16_bits(wl, 0)[0]
    xf = _bits_f32(xb)
    g, u, h = oracle.expert_gateup(wt, xf)
    Wg = _deq64(wt["gate_codes"], wt["gate_scales"])
    Wu = _deq64(wt["up_codes"], wt["up_scales"])
    x64 = xf.astype(np.float64)
    H = x64.size
    gamma = H * 2.0 ** -24 / (1 - H * 2.0 ** -24)
    for got, W in [(g, Wg), (u, Wu)]:
        ref = W @ x64
        bound = gamma * (np.abs(W) @ np.abs(x64))
        assert np.all(np.abs(got - ref) <= bound)
    # SwiGLU: torch's float64 silu of the oracle's own g, u; then bf16
    s64 = torch.nn.functional.silu(torch.from_numpy(g.astype(np.float64))).numpy() * u.astype(np.float64)
    h_ref = _bf16_bits(s64.astype(np.float32))
    diff = np.abs(h.astype(np.int32) - h_ref.astype(np.int32))
    assert np.all(diff <= 1) and np.mean(diff == 0) > 0.99


def _layer64(x_bits, ids, w, ws, prefill):
    """float64 evaluation of the layer; rounding steps via torch casts."""
    def mx8(bits_row_mat):
        x = torch.from_numpy(np.asarray(bits_row_mat, np.uint16).view(np.int16)).view(torch.bfloat16)
        xf = x.to(torch.float64).numpy()
        R, K = xf.shape
        blk = xf.reshape(R, K // 32, 32)
        amax = np.abs(blk).max(-1)
        _, ex = np.frexp(amax)
        sb = np.where(amax == 0, 0, np.clip(ex - 1 - 8 + 127, 0, 254)).astype(np.float64)
        sc = np.exp2(sb - 127)[..., None]
        q = torch.from_numpy(blk / sc).clamp(-448, 448).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        return (q * sc).reshape(R, K)

    T, H = x_bits.shape
    k = ids.shape[1]
    xin = mx8(x_bits) if prefill else _bits_f32(x_bits).astype(np.float64)
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            Wg = _deq64(ws["gate_codes"][e], ws["gate_scales"][e])
            Wu = _deq64(ws["up_codes"][e], ws["up_scales"][e])
            Wd = _deq64(ws["down_codes"][e], ws["down_scales"][e])
            g, u = Wg @ xin[t], Wu @ xin[t]
            hb = _bf16_bits((torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u).astype(np.float32))
            hin = mx8(hb[None, :])[0] if prefill else _bits_f32(hb).astype(np.float64)
            out[t] += float(w[t, j]) * (Wd @ hin)
    return out


@pytest.mark.parametrize("prefill", [False, True])
def test_layer_tiny_vs_float64(prefill):
    wl = S.WORKLOADS[0]
    ids, w = oracle.route(S.logits(wl, 0), wl.top_k)
    ws = S.stack_experts(S.layer_weights(wl, 0))
    x = S.activations_bf16_bits(wl, 0)
    out = oracle.layer(x, ids, w, ws, prefill=prefill, threads=4)
    ref = _layer64(x, ids, w, ws, prefill)
    rel = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    assert rel < 1e-4, rel
    # threads change nothing
    assert np.array_equal(out, oracle.layer(x, ids, w, ws, prefill=prefill, threads=1))


def test_layer_intermediates_consistent():
    wl = S.WORKLOADS[0]
    ids, w = oracle.route(S.logits(wl, 0), wl.top_k)
    ws = S.stack_experts(S.layer_weights(wl, 0))
    x = S.activations_bf16_bits(wl, 0)
    _, it = oracle.layer(x, ids, w, ws, prefill=True, want_intermediates=True)
    q, s = oracle.mxfp8_quant(x)
    assert np.array_equal(it["xq"], q) and np.array_equal(it["xs"], s)
    q2, s2 = oracle.mxfp8_quant(it["h"])
    assert np.array_equal(it["hq"], q2) and np.array_equal(it["hs"], s2)


_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _mx4_64(bits_rows):
    """MXFP4 quantise-dequantise in float64, written independently of the
    oracle: scale 2^(floor(log2 amax) - 2) per 32 (OCP MX v1.0 conversion
    with emax_elem = 2), each element the nearest E2M1 magnitude found by
    brute force over the 8 grid points, ties to the even code, sign kept."""
    x = _bits_f32(bits_rows).astype(np.float64)
    R, K = x.shape
    blk = x.reshape(R, K // 32, 32)
    amax = np.abs(blk).max(-1)
    _, ex = np.frexp(amax)
    sb = np.where(amax == 0, 0, np.clip(ex - 1 - 2 + 127, 0, 254)).astype(np.float64)
    sc = np.exp2(sb - 127)[..., None]
    a = np.abs(blk / sc)
    d = np.abs(a[..., None] - _E2M1_MAG)
    tie = d == d.min(-1, keepdims=True)
    even = tie & (np.arange(8) % 2 == 0)
    code = np.where(even.any(-1), even.argmax(-1), tie.argmax(-1))
    return (np.sign(blk) * _E2M1_MAG[code] * sc).reshape(R, K)


def _deq4_act(packed, scales):
    """Packed activation codes [R][K/2] + E8M0 [R][K/32] -> float64 [R][K]."""
    return _deq64(packed, scales)


def test_layer_mxfp4_activations_vs_float64():
    """The FP4-activation variant: both quantisation points reproduce the
    independent float64 MXFP4 quantiser exactly, h is the float64 SwiGLU to
    within one bf16 ulp, and out is the float64 down + combine of the
    quantised h within the fp32 summation bound."""
    wl = S.WORKLOADS[0]
    ids, w = oracle.route(S.logits(wl, 0), wl.top_k)
    ws = S.stack_experts(S.layer_weights(wl, 0))
    x = S.activations_bf16_bits(wl, 0)
    out, it = oracle.layer(x, ids, w, ws, prefill=True, act="mxfp4", want_intermediates=True, threads=4)
    T, H = x.shape
    k = ids.shape[1]
    I = ws["gate_codes"].shape[1]
    assert it["xq"].shape == (T, H // 2) and it["hq"].shape == (T * k, I // 2)
    xin = _mx4_64(x)
    assert np.array_equal(_deq4_act(it["xq"], it["xs"]), xin)
    # the same codes as the stand-alone quantiser
    q, sc = oracle.mxfp4_quant(x)
    assert np.array_equal(it["xq"], q) and np.array_equal(it["xs"], sc)
    hin = _mx4_64(it["h"])
    assert np.array_equal(_deq4_act(it["hq"], it["hs"]), hin)
    ref = np.zeros((T, H))
    bound = np.zeros((T, H))
    ulp = []
    for t in range(T):
        for j in range(k):
            e, a = ids[t, j], t * k + j
            Wg = _deq64(ws["gate_codes"][e], ws["gate_scales"][e])
            Wu = _deq64(ws["up_codes"][e], ws["up_scales"][e])
            Wd = _deq64(ws["down_codes"][e], ws["down_scales"][e])
            g, u = Wg @ xin[t], Wu @ xin[t]
            hb = _bf16_bits((torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u).astype(np.float32))
            ulp.append(np.abs(hb.astype(np.int32) - it["h"][a].astype(np.int32)))
            y = Wd @ hin[a]
            ref[t] += float(w[t, j]) * y
            bound[t] += abs(float(w[t, j])) * (np.abs(Wd) @ np.abs(hin[a]))
    ulp = np.concatenate(ulp)
    assert np.all(ulp <= 1) and np.mean(ulp == 0) > 0.99
    gamma = (I + k) * 2.0 ** -24 / (1 - (I + k) * 2.0 ** -24)
    assert np.all(np.abs(out - ref) <= gamma * bound + 1e-30)
    # threads change nothing; the FP8 mode is a different computation
    assert np.array_equal(out, oracle.layer(x, ids, w, ws, prefill=True, act="mxfp4", threads=1))
    assert not np.array_equal(out, oracle.layer(x, ids, w, ws, prefill=True, act="mxfp8"))


def test_layer_act_argument():
    wl = S.WORKLOADS[0]
    ids, w = oracle.route(S.logits(wl, 0), wl.top_k)
    ws = S.stack_experts(S.layer_weights(wl, 0))
    x = S.activations_bf16_bits(wl, 0)
    assert np.array_equal(oracle.layer(x, ids, w, ws, prefill=False),
                          oracle.layer(x, ids, w, ws, prefill=True, act="bf16"))
    assert np.array_equal(oracle.layer(x, ids, w, ws, prefill=True),
                          oracle.layer(x, ids, w, ws, prefill=False, act="mxfp8"))
    with pytest.raises(ValueError):
        oracle.layer(x, ids, w, ws, prefill=True, act="fp4")


def test_combine_pins():
    rng = np.random.default_rng(2)
    y = rng.standard_normal((5, 1, 64)).astype(np.float32)
    out = oracle.combine(y.reshape(5, 64), np.ones((5, 1), np.float32))
    assert np.array_equal(out, y[:, 0])
    y = rng.standard_normal((5 * 3, 64)).astype(np.float32)
    w = rng.random((5, 3)).astype(np.float32)
    out = oracle.combine(y, w)
    ref = np.einsum("tj,tjh->th", w.astype(np.float64), y.reshape(5, 3, 64).astype(np.float64))
    assert np.max(np.abs(out - ref)) <= 4 * 2.0 ** -24 * np.max(np.abs(ref)) * 3
    # order matters only through rounding: swapping j changes nothing exactly here
    assert np.allclose(out, ref, rtol=1e-6, atol=1e-6)
