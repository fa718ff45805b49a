"""Seeded synthetic inputs for the routed-expert FFN layer.

This module only *draws* inputs: router logits, bf16 activations and MXFP4
expert weights in the canonical byte layout. It holds none of the layer's
arithmetic (no top-k, no softmax, no dequantisation, no matmul), so both the
CPU oracle and the CUDA path can read the same buffers without sharing any
code of the method.

Workload shapes follow the two model families the tinyserve README and the
llama.cpp fixed-expert-pool discussion benchmark: a GPT-OSS-20B-shaped layer
(hidden 2880, expert intermediate 2880, 32 experts, top-4, 24 layers) and a
Qwen-30B-A3B-shaped layer (hidden 2048, intermediate 768, 128 experts, top-8).

Every tensor has its own PCG64 stream keyed by
``[SEED, workload id, tensor tag, layer, index]`` so generation order never
matters and any single expert can be regenerated on its own.

Canonical MXFP4 layout (one matrix of ``rows x K``):
  * codes  : uint8 ``[rows][K/2]``, element ``2i`` in the low nibble of byte ``i``;
  * scales : uint8 ``[rows][K/32]`` E8M0 bytes, one per 32-element block along K.
Gate and up are ``[I][H]``; down is ``[H][I]``.

GGUF weights (``gguf_matrix``) are rows of Q8_0 blocks (32 elements in 34
bytes) or Q4_K super-blocks (256 elements in 144 bytes) along K, drawn as
random bytes with their binary16 scales set to a bounded range.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass

import numpy as np

SEED = 0

TAG_LOGITS = 1
TAG_RANK = 2
TAG_X = 3
TAG_GATE = 4
TAG_UP = 5
TAG_DOWN = 6

TAG_GGUF = 16       # + 0 gate, 1 up, 2 down; GGUF block streams

# E8M0 scale bytes are 127 + e with e uniform in {-6,...,-2}.
SCALE_BYTE_LO = 121
SCALE_BYTE_SPAN = 5


@dataclass(frozen=True)
class Workload:
    """Shape and routing recipe of one synthetic workload."""

    wid: int            # workload id; keys the random streams
    name: str
    layers: int         # L
    hidden: int         # H
    inter: int          # I (expert intermediate)
    experts: int        # E
    top_k: int          # k
    tokens: int         # T per layer call
    steps: int          # decode steps (1 for prefill / tiny)
    slots: int          # GPU expert slots per layer (S); S == E means resident
    bias_c: float       # logits += -bias_c * ln(rank_e); 0 disables
    weight_wid: int     # workload id whose weight streams are reused

    @property
    def resident(self) -> bool:
        return self.slots == self.experts


WORKLOADS = {
    0: Workload(0, "tiny_h256_i512_e8_k2_t16", 1, 256, 512, 8, 2, 16, 1, 8, 0.0, 0),
    1: Workload(1, "gptoss20b_decode_resident_l24_h2880_e32_k4", 24, 2880, 2880, 32, 4, 1, 256, 32, 0.0, 1),
    2: Workload(2, "gptoss20b_decode_offload_s8_lru", 24, 2880, 2880, 32, 4, 1, 256, 8, 1.2, 1),
    3: Workload(3, "gptoss20b_prefill_t3072", 1, 2880, 2880, 32, 4, 3072, 1, 32, 0.0, 3),
    4: Workload(4, "qwen30b_a3b_prefill_t16384", 1, 2048, 768, 128, 8, 16384, 1, 128, 0.8, 4),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng([SEED, *[int(k) for k in key]])


def expert_rank(wl: Workload, layer: int) -> np.ndarray:
    """Seeded permutation of 1..E per layer (the rank used by the routing skew)."""
    return _rng(wl.wid, TAG_RANK, layer).permutation(wl.experts).astype(np.int64) + 1


def logits(wl: Workload, layer: int, step: int = 0, tokens: int | None = None) -> np.ndarray:
    """Router logits, fp32 ``[T, E]``: N(0,1), plus ``-c*ln(rank_e)`` when skewed.

    The bias is evaluated in float64, rounded to fp32 and added in fp32, so
    every consumer sees identical logits.
    """
    T = wl.tokens if tokens is None else tokens
    z = _rng(wl.wid, TAG_LOGITS, layer, step).standard_normal((T, wl.experts), dtype=np.float32)
    if wl.bias_c:
        bias = (-wl.bias_c * np.log(expert_rank(wl, layer).astype(np.float64))).astype(np.float32)
        z = (z + bias[None, :]).astype(np.float32)
    return np.ascontiguousarray(z)


def activations_f32(wl: Workload, layer: int, step: int = 0, tokens: int | None = None) -> np.ndarray:
    """N(0,1) fp32 draws that become the bf16 activations ``[T, H]``."""
    T = wl.tokens if tokens is None else tokens
    return _rng(wl.wid, TAG_X, layer, step).standard_normal((T, wl.hidden), dtype=np.float32)


def activations_bf16_bits(wl: Workload, layer: int, step: int = 0, tokens: int | None = None) -> np.ndarray:
    """bf16 activations ``[T, H]`` as uint16 bit patterns (torch's RNE cast)."""
    import torch

    x = torch.from_numpy(activations_f32(wl, layer, step, tokens)).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16).copy()


def _matrix(wl: Workload, tag: int, layer: int, expert: int, rows: int, K: int):
    rng = _rng(wl.weight_wid, tag, layer, expert)
    codes = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    scales = (SCALE_BYTE_LO + rng.integers(0, SCALE_BYTE_SPAN, size=(rows, K // 32), dtype=np.uint8)).astype(np.uint8)
    return codes, scales


def expert_weights(wl: Workload, layer: int, expert: int) -> dict:
    """Canonical MXFP4 weights of one expert (gate/up ``[I][H]``, down ``[H][I]``)."""
    H, I = wl.hidden, wl.inter
    gc, gs = _matrix(wl, TAG_GATE, layer, expert, I, H)
    uc, us = _matrix(wl, TAG_UP, layer, expert, I, H)
    dc, ds = _matrix(wl, TAG_DOWN, layer, expert, H, I)
    return dict(gate_codes=gc, gate_scales=gs, up_codes=uc, up_scales=us,
                down_codes=dc, down_scales=ds)


GGUF_BLOCK = {"q8_0": (32, 34), "q4_k": (256, 144)}   # elements, bytes per block


def gguf_matrix(wl: Workload, fmt: str, which: int, layer: int, expert: int, rows: int, K: int) -> np.ndarray:
    """GGUF block bytes ``[rows, K/n * bytes]`` of one matrix (``which``: 0
    gate, 1 up, 2 down), random in every byte except the binary16 scales:
    Q8_0 ``d`` and Q4_K ``d``/``dmin`` are 2^u with u uniform in [-9, -6)
    (Q8_0) or [-9, -7) (Q4_K), rounded to binary16, little-endian.  The
    6-bit scales/mins and the values are uniform over their codes."""
    n, nbytes = GGUF_BLOCK[fmt]
    if K % n:
        raise ValueError(f"K={K} is not a multiple of {n} ({fmt})")
    rng = _rng(wl.weight_wid, TAG_GGUF + which, layer, expert, nbytes)
    nb = K // n
    blk = rng.integers(0, 256, size=(rows, nb, nbytes), dtype=np.uint8)
    if fmt == "q8_0":
        d = np.exp2(rng.uniform(-9, -6, size=(rows, nb))).astype("<f2")
        blk[..., 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    else:
        d = np.exp2(rng.uniform(-9, -7, size=(rows, nb, 2))).astype("<f2")
        blk[..., 0:4] = d.view(np.uint8).reshape(rows, nb, 4)
    return blk.reshape(rows, nb * nbytes)


def expert_weights_gguf(wl: Workload, fmt: str, layer: int, expert: int) -> dict:
    """GGUF weights of one expert: ``gate``/``up`` ``[I][row bytes of H]``,
    ``down`` ``[H][row bytes of I]``."""
    H, I = wl.hidden, wl.inter
    return dict(gate=gguf_matrix(wl, fmt, 0, layer, expert, I, H),
                up=gguf_matrix(wl, fmt, 1, layer, expert, I, H),
                down=gguf_matrix(wl, fmt, 2, layer, expert, H, I))


def layer_weights(wl: Workload, layer: int, experts=None, threads: int | None = None) -> list:
    """Weights of several experts of one layer, drawn in parallel threads.

    numpy's generators release the GIL while filling large arrays, and each
    expert has an independent stream, so the result does not depend on the
    thread count.
    """
    ids = list(range(wl.experts)) if experts is None else list(experts)
    threads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda e: expert_weights(wl, layer, e), ids))


def stack_experts(ws: list) -> dict:
    """Stack a list of per-expert dicts into ``[E, ...]`` arrays."""
    return {k: np.ascontiguousarray(np.stack([w[k] for w in ws])) for k in ws[0]}
