"""Shared test plumbing: building pools from the seeded workloads and
comparing results.  Imports the oracle (tests may) and the product binding."""
from __future__ import annotations

import numpy as np

import moe_synth as S

ULP_TOL_W = 2  # routing weights: |delta| <= 2 ulp


def f32_ulp_diff(a, b):
    """Distance in units in the last place between fp32 arrays."""
    ai = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ai = np.where(ai < 0, np.int64(-2 ** 31) - ai, ai)
    bi = np.where(bi < 0, np.int64(-2 ** 31) - bi, bi)
    return np.abs(ai - bi)


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def build_host_store(M, wl, layers=None, experts=None, threads=16):
    """Pinned host tensor [L][E][expert_bytes] of packed experts (moe_pack_expert)."""
    import torch

    L = wl.layers if layers is None else layers
    E = wl.experts
    eb = M.moe_expert_bytes(wl.hidden, wl.inter)
    host = torch.empty(L * E * eb, dtype=torch.uint8).pin_memory()
    base = host.data_ptr()
    exps = list(range(E)) if experts is None else list(experts)
    for l in range(L):
        ws = S.layer_weights(wl, l, exps, threads=threads)
        for e, w in zip(exps, ws):
            M.moe_pack_expert(w, wl.hidden, wl.inter, base + (l * E + e) * eb)
    return host, eb


def make_pool(M, wl, layers=None, slots=None, preload=True, device="cuda"):
    import torch

    L = wl.layers if layers is None else layers
    S_ = wl.slots if slots is None else slots
    host, eb = build_host_store(M, wl, L)
    dev = torch.empty(L * S_ * eb, dtype=torch.uint8, device=device)
    pool = M.Pool(L, wl.experts, S_, wl.hidden, wl.inter, host_experts=host, dev_slots=dev, preload=preload)
    return pool, host, dev
