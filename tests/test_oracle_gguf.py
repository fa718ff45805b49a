"""Pins of the oracle's GGUF block formats (Q8_0, Q4_K) and of its decode
layer on GGUF expert weights.

The tinyserve README ("How it works" item 2; "Supported models", Formats)
names Q4_K, Q5_K, Q6_K and Q8_0 as the GGUF formats it computes on without
a dequantised copy; the block layouts are the published GGUF / ggml ones.
What pins them here: binary16 against torch over every bit pattern;
hand-worked blocks (``tests/golden/gguf_*.txt``); one-hot super-blocks
that locate every element's nibble; the full range of 6-bit scales and
mins; and a cross-format identity: on weights that MXFP4 and a GGUF format
both represent exactly, the GGUF decode layer equals the (separately
pinned) MXFP4 decode layer bit for bit."""
import os

import numpy as np
import pytest
import torch

import moe_synth as S
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def _lines(name):
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            yield line


def test_f16_every_code_vs_torch():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.float16).double().numpy()
    got = np.array([oracle.f16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_row_bytes():
    assert oracle.gguf_row_bytes("q8_0", 2880) == 90 * 34
    assert oracle.gguf_row_bytes("q4_k", 2048) == 8 * 144
    assert oracle.gguf_row_bytes("q4_k", 768) == 3 * 144
    assert oracle.gguf_row_bytes("q4_k", 2880) == 0      # not a multiple of 256
    assert oracle.gguf_row_bytes("q8_0", 48) == 0
    with pytest.raises(ValueError):
        oracle.dequant_gguf("q4_k", np.zeros((1, 144), np.uint8), 2880)


def test_q8_0_hand_worked_blocks():
    for line in _lines("gguf_q8_0_blocks.txt"):
        d_hex, q_txt, v_txt = (f.strip() for f in line.split("|"))
        q = np.array([int(v) for v in q_txt.split()], np.int8)
        want = np.array([float(v) for v in v_txt.split()], np.float32)
        blk = np.zeros((1, 34), np.uint8)
        d = int(d_hex, 16)
        blk[0, 0], blk[0, 1] = d & 0xFF, d >> 8
        blk[0, 2:] = q.view(np.uint8)
        got = oracle.dequant_gguf("q8_0", blk, 32)[0]
        assert np.array_equal(got, want), (d_hex, got)


def test_q8_0_random_rows_vs_numpy_f16():
    rng = np.random.default_rng(7)
    rows, K = 16, 320
    b = rng.integers(0, 256, size=(rows, K // 32, 34), dtype=np.uint8)
    d = b[..., 0:2].copy().view("<f2")[..., 0].astype(np.float64)          # any binary16, inf/NaN included
    q = b[..., 2:].view(np.int8).astype(np.float64)
    with np.errstate(invalid="ignore"):
        want = (d[..., None] * q).astype(np.float32).reshape(rows, K)
    got = oracle.dequant_gguf("q8_0", b.reshape(rows, -1), K)
    both_nan = np.isnan(want) & np.isnan(got)
    assert np.array_equal(got[~both_nan], want[~both_nan])


def _q4_k_golden():
    f = {}
    sc_m, vals = {}, {}
    for line in _lines("gguf_q4_k_superblock.txt"):
        key, *rest = line.split()
        if key == "sc_m":
            sc_m[int(rest[0])] = (int(rest[1]), int(rest[2]))
        elif key == "values":
            vals[int(rest[0])] = np.array([float(v) for v in rest[1:]])
        else:
            f[key] = rest
    blk = np.zeros(144, np.uint8)
    for off, key in [(0, "d"), (2, "dmin")]:
        v = int(f[key][0], 16)
        blk[off], blk[off + 1] = v & 0xFF, v >> 8
    blk[4:16] = [int(x, 16) for x in f["p"]]
    l = np.arange(32)
    for g in range(4):
        blk[16 + 32 * g:16 + 32 * g + 32] = (l & 15) | ((15 - (l & 15)) << 4)
    return blk, sc_m, vals


def test_q4_k_hand_worked_superblock():
    blk, sc_m, vals = _q4_k_golden()
    got = oracle.dequant_gguf("q4_k", blk[None, :], 256)[0].reshape(8, 32)
    l = np.arange(32)
    for j in range(8):
        sc, m = sc_m[j]
        q = (l & 15) if j % 2 == 0 else 15 - (l & 15)
        assert np.array_equal(got[j], (1.0 * sc * q - 0.5 * m).astype(np.float32)), j
        if j in vals:
            assert np.array_equal(got[j, :16], vals[j].astype(np.float32))
            assert np.array_equal(got[j, 16:], vals[j].astype(np.float32))


def _pack_q4_k(d_bits, dmin_bits, sc, m, q):
    """One super-block from its fields (the inverse of the layout the
    oracle reads, written from the same published description)."""
    blk = np.zeros(144, np.uint8)
    blk[0:2] = [d_bits & 0xFF, d_bits >> 8]
    blk[2:4] = [dmin_bits & 0xFF, dmin_bits >> 8]
    p = np.zeros(12, np.int64)
    for j in range(4):
        p[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        p[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        p[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    blk[4:16] = p
    q = np.asarray(q).reshape(8, 32)
    for g in range(4):
        blk[16 + 32 * g:48 + 32 * g] = q[2 * g] | (q[2 * g + 1] << 4)
    return blk


def test_q4_k_one_hot_locates_every_element():
    """256 super-blocks, the n-th with q = 15 at element n and 0 elsewhere,
    scale 1, min 0: exactly element n is 15."""
    blocks = np.stack([_pack_q4_k(0x3C00, 0x3C00, [1] * 8, [0] * 8, np.eye(256, dtype=np.int64)[n] * 15)
                       for n in range(256)])
    got = oracle.dequant_gguf("q4_k", blocks.reshape(256, 144), 256)
    assert np.array_equal(got, 15 * np.eye(256, dtype=np.float32))


def test_q4_k_every_scale_and_min_code():
    """All 64 codes of sc and of m, in every sub-block position (4 of the
    8 use the split 4+2-bit packing)."""
    rng = np.random.default_rng(3)
    blocks, want = [], []
    for rot in range(64):
        sc = [(rot + 8 * j) % 64 for j in range(8)]
        m = [(rot * 5 + 3 * j + 11) % 64 for j in range(8)]
        q = rng.integers(0, 16, 256)
        blocks.append(_pack_q4_k(0x3400, 0x2C00, sc, m, q))          # d = 0.25, dmin = 0.0625
        want.append((0.25 * np.repeat(sc, 32) * q - 0.0625 * np.repeat(m, 32)).astype(np.float32))
    got = oracle.dequant_gguf("q4_k", np.stack(blocks), 256)
    assert np.array_equal(got, np.stack(want))


def test_q4_k_random_rows_single_rounding():
    """Random super-blocks (the synthetic generator's): each element is the
    fp32 rounding of the exact d*sc*q - dmin*m (float64 holds it exactly
    for these exponents)."""
    wl = S.WORKLOADS[0]
    b = S.gguf_matrix(wl, "q4_k", 0, 0, 0, 8, 512).reshape(8, 2, 144)
    got = oracle.dequant_gguf("q4_k", b.reshape(8, -1), 512).reshape(8, 2, 8, 32)
    d = b[..., 0:2].copy().view("<f2")[..., 0].astype(np.float64)
    dmin = b[..., 2:4].copy().view("<f2")[..., 0].astype(np.float64)
    p = b[..., 4:16].astype(np.int64)
    sc = np.concatenate([p[..., 0:4] & 63, (p[..., 8:12] & 15) | ((p[..., 0:4] >> 6) << 4)], -1)
    m = np.concatenate([p[..., 4:8] & 63, (p[..., 8:12] >> 4) | ((p[..., 4:8] >> 6) << 4)], -1)
    qs = b[..., 16:].reshape(8, 2, 4, 32).astype(np.int64)
    q = np.stack([qs & 15, qs >> 4], 3).reshape(8, 2, 8, 32)
    exact = d[..., None, None] * sc[..., None] * q - dmin[..., None, None] * m[..., None]
    assert np.array_equal(got, exact.astype(np.float32))


# ---- the decode layer on GGUF weights ---------------------------------------

def _mxfp4_values(codes, scales):
    lo, hi = codes & 15, codes >> 4
    el = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.int64)
    el[..., 0::2] = lo
    el[..., 1::2] = hi
    return el, scales.astype(np.int64)


def _q8_0_from_mxfp4(codes, scales):
    """MXFP4 rows -> Q8_0 rows holding the same values: per 32-block
    d = 2^(s-128) (binary16 holds it for s >= 104), q = 2 * E2M1 value."""
    el, sc = _mxfp4_values(codes, scales)
    rows, K = el.shape
    assert sc.min() >= 104
    out = np.zeros((rows, K // 32, 34), np.uint8)
    d = np.exp2(sc - 128.0).astype("<f2")
    out[..., 0:2] = d.view(np.uint8).reshape(rows, K // 32, 2)
    q = (2 * E2M1[el]).astype(np.int8).reshape(rows, K // 32, 32)
    out[..., 2:] = q.view(np.uint8)
    return out.reshape(rows, -1)


def _q4_k_mxfp4_pair(rng, rows, K):
    """Weights both formats hold exactly: per super-block d = dmin = 2^-8;
    per sub-block sc in {1, 2, 4}; a sub-block of non-negative E2M1 values
    uses m = 0 and q = 2v/sc', one of non-positive values m = 12 sc and
    q = 12 + 2v/sc' (sc' = 2^(-8) sc scaling, v the E2M1 magnitude grid).
    Returns (Q4_K rows, MXFP4 codes, MXFP4 scales)."""
    nb = K // 256
    q4 = np.zeros((rows, nb, 144), np.uint8)
    codes = np.zeros((rows, K // 2), np.uint8)
    scales = np.zeros((rows, K // 32), np.uint8)
    for r in range(rows):
        for b in range(nb):
            sc = rng.choice([1, 2, 4], 8)
            neg = rng.integers(0, 2, 8).astype(bool)
            m = np.where(neg, 12 * sc, 0)
            mag = rng.integers(0, 8, (8, 32))                  # E2M1 magnitude code
            twice = (2 * E2M1[mag]).astype(np.int64)           # 0 1 2 3 4 6 8 12
            q = np.where(neg[:, None], 12 - twice, twice)
            q4[r, b] = _pack_q4_k(0x1C00, 0x1C00, sc, m, q)   # 2^-8
            # value = 2^-8 * sc * (+-twice) = E2M1(+-mag) * 2^(-7) * sc
            code = np.where(neg[:, None] & (mag > 0), mag | 8, mag)
            for j in range(8):
                c = (b * 8 + j) * 32
                scales[r, c // 32] = 127 - 7 + int(np.log2(sc[j]))
                blk = code[j]
                codes[r, c // 2:c // 2 + 16] = blk[0::2] | (blk[1::2] << 4)
    return q4.reshape(rows, -1), codes, scales


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_layer_gguf_equals_mxfp4_layer_on_shared_values(fmt):
    wl = S.WORKLOADS[0]
    ids, w = oracle.route(S.logits(wl, 0), wl.top_k)
    x = S.activations_bf16_bits(wl, 0)
    H, I = wl.hidden, wl.inter
    if fmt == "q8_0":
        mx = S.stack_experts(S.layer_weights(wl, 0))
        gg = {}
        for name, key in [("gate", "gate"), ("up", "up"), ("down", "down")]:
            gg[name] = np.stack([_q8_0_from_mxfp4(mx[key + "_codes"][e], mx[key + "_scales"][e])
                                 for e in range(wl.experts)])
    else:
        rng = np.random.default_rng(5)
        mx, gg = {}, {}
        for name, rows, K in [("gate", I, H), ("up", I, H), ("down", H, I)]:
            parts = [_q4_k_mxfp4_pair(rng, rows, K) for _ in range(wl.experts)]
            gg[name] = np.stack([p[0] for p in parts])
            mx[name + "_codes"] = np.stack([p[1] for p in parts])
            mx[name + "_scales"] = np.stack([p[2] for p in parts])
        # the constructed pair really holds the same values
        assert np.array_equal(oracle.dequant_gguf("q4_k", gg["down"][0], I),
                              oracle.dequant_mxfp4(mx["down_codes"][0], mx["down_scales"][0]))
    ref = oracle.layer(x, ids, w, mx, prefill=False, threads=4)
    out, h = oracle.layer_gguf(fmt, x, ids, w, gg, threads=4, want_h=True)
    assert np.array_equal(out, ref)
    assert np.array_equal(out, oracle.layer_gguf(fmt, x, ids, w, gg, threads=1))


def _bits_f32(b):
    return torch.from_numpy(np.asarray(b, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


def _bf16_bits(f):
    return torch.from_numpy(np.asarray(f, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_layer_gguf_vs_float64(fmt):
    """Synthetic GGUF weights: h within one bf16 ulp of the float64 SwiGLU
    of float64 sums over the oracle's own dequantised weights, out within
    the fp32 summation bound of the float64 down + combine of the oracle's
    h.  Where g < -88.7 the fp32 exp(-g) of silu overflows and silu(g) is
    -0 (the biased Q4_K draws reach that): for g < -87 both hs are below
    1e-30 and only that is checked."""
    wl = S.WORKLOADS[0]
    ids, w = oracle.route(S.logits(wl, 0), wl.top_k)
    x = S.activations_bf16_bits(wl, 0)
    H, I, k = wl.hidden, wl.inter, wl.top_k
    ws = [S.expert_weights_gguf(wl, fmt, 0, e) for e in range(wl.experts)]
    gg = {n: np.stack([e[n] for e in ws]) for n in ("gate", "up", "down")}
    out, h = oracle.layer_gguf(fmt, x, ids, w, gg, threads=4, want_h=True)
    xf = _bits_f32(x).astype(np.float64)
    ref = np.zeros(out.shape)
    bound = np.zeros(out.shape)
    ulp = []
    for t in range(x.shape[0]):
        for j in range(k):
            e, a = ids[t, j], t * k + j
            Wg = oracle.dequant_gguf(fmt, gg["gate"][e], H).astype(np.float64)
            Wu = oracle.dequant_gguf(fmt, gg["up"][e], H).astype(np.float64)
            Wd = oracle.dequant_gguf(fmt, gg["down"][e], I).astype(np.float64)
            g, u = Wg @ xf[t], Wu @ xf[t]
            hb = _bf16_bits((torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u).astype(np.float32))
            tiny = (g < -87) | (np.abs(_bits_f32(hb)) < 2.0 ** -126)
            assert np.all(np.abs(_bits_f32(h[a])[tiny]) <= 1e-30)
            ulp.append(np.abs(hb.astype(np.int32) - h[a].astype(np.int32))[~tiny])
            hin = _bits_f32(h[a]).astype(np.float64)
            ref[t] += float(w[t, j]) * (Wd @ hin)
            bound[t] += abs(float(w[t, j])) * (np.abs(Wd) @ np.abs(hin))
    ulp = np.concatenate(ulp)
    assert np.all(ulp <= 1) and np.mean(ulp == 0) > 0.99
    gamma = (I + k) * 2.0 ** -24 / (1 - (I + k) * 2.0 ** -24)
    assert np.all(np.abs(out - ref) <= gamma * bound + 1e-30)


def test_layer_gguf_rejects_bad_shapes():
    wl = S.WORKLOADS[0]
    ids, w = oracle.route(S.logits(wl, 0), wl.top_k)
    x = S.activations_bf16_bits(wl, 0)
    ws = [S.expert_weights_gguf(wl, "q8_0", 0, e) for e in range(wl.experts)]
    gg = {n: np.stack([e[n] for e in ws]) for n in ("gate", "up", "down")}
    with pytest.raises(ValueError):
        oracle.layer_gguf("q4_k", x, ids, w, gg)           # q8_0 bytes read as q4_k
    bad = ids.copy()
    bad[0, 0] = wl.experts
    with pytest.raises(ValueError):
        oracle.layer_gguf("q8_0", x, bad, w, gg)
