"""Pins of the oracle's number formats against the OCP specifications' tables
and torch's own casts (library routines independent of the oracle)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _table(name):
    rows = []
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            a, b = line.split()
            rows.append((int(a, 0), float(b)))
    return rows


def test_e2m1_matches_ocp_table():
    for code, val in _table("e2m1_table.txt"):
        got = oracle.e2m1_value(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got, val)


def test_e8m0_closed_form():
    for b in range(255):
        assert oracle.e8m0_value(b) == 2.0 ** (b - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_e4m3_named_points():
    for code, val in _table("e4m3_points.txt"):
        got = oracle.e4m3_value(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val)
        assert oracle.e4m3_encode(val) == code
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def test_e4m3_decode_all_codes_vs_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], c


def test_e4m3_encode_every_inrange_bf16_vs_torch():
    """Every finite bf16 pattern with |v| <= 448: RNE must agree with torch's cast."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    keep = torch.isfinite(vals) & (vals.abs() <= 448)
    vals = vals[keep]
    ref = vals.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    v64 = vals.to(torch.float64).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in v64], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(v64[i], got[i], ref[i]) for i in bad[:5]]


def test_e4m3_saturates_to_448():
    for v in [448.0, 449.0, 463.9, 464.0, 480.0, 511.0, 1e6, float("inf")]:
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE


def test_bf16_rne_vs_torch():
    rng = np.random.default_rng(7)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(2000) * 1e-38).astype(np.float32),
                        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.4e38, 1e-45], np.float32)])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(x)) for x in f], np.uint16)
    assert np.array_equal(got, ref)
    for b in [0x3F80, 0xBF80, 0x0001, 0x7F7F]:
        ref_f = torch.from_numpy(np.array([b], np.uint16).view(np.int16)).view(torch.bfloat16).float().item()
        assert oracle.bf16_to_f32(b) == ref_f


def _parse_blocks():
    out = []
    for line in open(os.path.join(GOLD, "mxfp8_blocks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, sb, codes = line.split("|")
        name, *vals = head.split()
        out.append((name, [float(v) for v in vals], int(sb), [int(c, 16) for c in codes.split()]))
    return out


def test_mxfp8_hand_worked_blocks():
    for name, vals, sb, codes in _parse_blocks():
        x = torch.tensor(vals, dtype=torch.float64)
        xb = x.to(torch.bfloat16)
        assert torch.equal(xb.to(torch.float64), x), name  # fixtures are exact bf16
        q, s = oracle.mxfp8_quant(xb.view(torch.int16).numpy().view(np.uint16)[None, :])
        assert s[0, 0] == sb, (name, s[0, 0], sb)
        assert q[0].tolist() == codes, (name, q[0].tolist())


def test_mxfp8_random_vs_torch_cast():
    """Scale from the exponent of amax (numpy frexp); elements from torch's
    e4m3fn cast of x / scale after clamping to +-448 (satfinite)."""
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((64, 256)).astype(np.float32) * 3).to(torch.bfloat16)
    x[5, :32] = 0
    x[6, 32:64] = torch.tensor(1e-30)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.mxfp8_quant(bits)
    xf = x.to(torch.float64).numpy().reshape(64, 8, 32)
    amax = np.abs(xf).max(-1)
    _, ex = np.frexp(amax)
    sb_ref = np.where(amax == 0, 0, np.clip(ex - 1 - 8 + 127, 0, 254))
    assert np.array_equal(s, sb_ref.astype(np.uint8))
    scaled = torch.from_numpy(xf / np.exp2(sb_ref.astype(np.float64) - 127)[..., None])
    q_ref = scaled.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(64, 256)
    assert np.array_equal(q, q_ref)


def test_dequant_mxfp4_against_table():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 256, (8, 64), dtype=np.uint8)
    scales = (118 + rng.integers(0, 12, (8, 4))).astype(np.uint8)
    tab = np.array([v for _, v in _table("e2m1_table.txt")])
    lo, hi = codes & 15, codes >> 4
    el = np.empty((8, 128), np.float64)
    el[:, 0::2] = tab[lo]
    el[:, 1::2] = tab[hi]
    ref = el * np.exp2(np.repeat(scales.astype(np.float64) - 127, 32, axis=1))
    got = oracle.dequant_mxfp4(codes, scales)
    assert np.array_equal(got.astype(np.float64), ref)


def _e2m1_nearest(v):
    """Brute force: the E2M1 code whose value is nearest to v, ties to the
    code with mantissa bit 0, sign kept (including for zero)."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    a = abs(v)
    best = min(range(8), key=lambda i: (abs(a - mags[i]), i & 1))
    return best | (8 if math.copysign(1.0, v) < 0 else 0)


def test_e2m1_encode_hand_worked_cases():
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "e2m1_rounding.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        v, code = line.split()
        assert oracle.e2m1_encode(float(v)) == int(code), v


def test_e2m1_encode_matches_brute_force_nearest():
    rng = np.random.default_rng(4)
    vals = list(rng.standard_normal(20000) * 3) + list(rng.uniform(-8, 8, 20000))
    vals += [m / 4 for m in range(-40, 41)]          # every quarter step: all ties
    for v in vals:
        assert oracle.e2m1_encode(float(v)) == _e2m1_nearest(float(v)), v
    for c in range(16):                              # the grid maps to itself
        assert oracle.e2m1_encode(oracle.e2m1_value(c)) == c


def test_mxfp4_quant_scale_rule_and_bound():
    """Scale byte = floor(log2 amax) - 2 + 127 (OCP MX v1.0 6.3, emax 2 for
    E2M1); every element dequantises to within half the local grid step or
    saturates to 6 * scale; zero blocks give scale 0 and zero codes."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((8, 256)) * np.exp(rng.uniform(-8, 8, (8, 1)))).astype(np.float32)
    x[3, 64:96] = 0.0
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.mxfp4_quant(bits)
    xf = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    for r in range(8):
        for b in range(256 // 32):
            blk = xf[r, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            if amax == 0:
                assert s[r, b] == 0 and not q[r, 16 * b:16 * b + 16].any()
                continue
            assert s[r, b] == math.frexp(amax)[1] - 1 - 2 + 127
            scale = 2.0 ** (int(s[r, b]) - 127)
            for i in range(32):
                byte = q[r, 16 * b + i // 2]
                code = (byte >> 4) if i & 1 else (byte & 15)
                got = oracle.e2m1_value(code) * scale
                ref = blk[i]
                if abs(ref) / scale >= 6.0:
                    assert got == math.copysign(6.0 * scale, ref)
                else:
                    a = abs(ref) / scale                      # grid steps 0.5 / 1 / 2 below 2 / 4 / 6
                    half_step = 0.25 if a < 2 else (0.5 if a < 4 else 1.0)
                    assert abs(got - ref) <= half_step * scale
