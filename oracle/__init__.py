"""CPU oracle of the routed-expert FFN layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports it and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain C, compiled with gcc,
``-O2 -ffp-contract=off``, no fast-math); this module only marshals numpy
arrays through ctypes.  Every function names the passage it follows in the C
source.

Parity status per function (what pins it, see ``tests/test_oracle_*.py``):
  * e2m1/e8m0/e4m3/bf16 codecs ........ pinned (OCP spec table, torch casts)
  * mxfp8_quant_row ................... pinned (torch e4m3 cast, frexp, closed form)
  * route (top-k + softmax) ........... pinned (brute-force sort, closed forms)
  * hist_perm ......................... pinned (numpy stable argsort, invariants)
  * lru_step .......................... pinned (independent list simulator, hand cases)
  * expert_gateup / expert_down ....... pinned (integer-exact case, float64 numpy bound)
  * layer (decode, prefill) ........... pinned piecewise; the end-to-end float
                                        value has no printed worked example
  * combine ........................... pinned (k=1 identity, float64 bound)
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_INVALID = -1
ERR_CAPACITY = -3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build`` (if stale)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            vp, i32, i64p = C.c_void_p, C.c_int, C.POINTER(C.c_int64)
            L.oracle_e2m1_value.restype = C.c_double
            L.oracle_e2m1_value.argtypes = [C.c_uint8]
            L.oracle_e8m0_value.restype = C.c_double
            L.oracle_e8m0_value.argtypes = [C.c_uint8]
            L.oracle_e4m3_value.restype = C.c_double
            L.oracle_e4m3_value.argtypes = [C.c_uint8]
            L.oracle_e4m3_encode.restype = C.c_uint8
            L.oracle_e4m3_encode.argtypes = [C.c_double]
            L.oracle_bf16_to_f32.restype = C.c_float
            L.oracle_bf16_to_f32.argtypes = [C.c_uint16]
            L.oracle_f32_to_bf16.restype = C.c_uint16
            L.oracle_f32_to_bf16.argtypes = [C.c_float]
            L.oracle_mxfp8_quant_row.argtypes = [vp, i32, vp, vp]
            L.oracle_dequant_mxfp4.argtypes = [vp, vp, i32, i32, vp]
            L.oracle_route.argtypes = [vp, i32, i32, i32, vp, vp]
            L.oracle_hist_perm.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
            L.oracle_lru_step.argtypes = [i32, i32, vp, vp, vp, vp, i64p, i64p, i64p, i64p, vp, vp, vp]
            L.oracle_expert_gateup.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp]
            L.oracle_expert_down.argtypes = [vp, vp, i32, i32, vp, vp]
            L.oracle_layer.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                       vp, vp, vp, vp, vp, vp, i32]
            L.oracle_combine.argtypes = [vp, vp, i32, i32, i32, vp]
            _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- formats ---------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def e8m0_value(b: int) -> float:
    return lib().oracle_e8m0_value(b)


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(code)


def e4m3_encode(v: float) -> int:
    return lib().oracle_e4m3_encode(v)


def bf16_to_f32(b: int) -> float:
    return lib().oracle_bf16_to_f32(b)


def f32_to_bf16(f: float) -> int:
    return lib().oracle_f32_to_bf16(f)


def mxfp8_quant(x_bf16_bits: np.ndarray):
    """MXFP8 of each row of ``[rows, K]`` bf16 bits -> (codes u8, scales u8)."""
    x = _c(x_bf16_bits, np.uint16)
    rows, K = x.shape
    q = np.zeros((rows, K), np.uint8)
    s = np.zeros((rows, K // 32), np.uint8)
    for r in range(rows):
        lib().oracle_mxfp8_quant_row(_p(x[r]), K, _p(q[r]), _p(s[r]))
    return q, s


def dequant_mxfp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows, K = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((rows, K), np.float32)
    lib().oracle_dequant_mxfp4(_p(codes), _p(scales), rows, K, _p(out))
    return out


# ---- routing ---------------------------------------------------------------

def route(logits: np.ndarray, k: int):
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    rc = lib().oracle_route(_p(lg), T, E, k, _p(ids), _p(w))
    if rc != OK:
        raise ValueError(f"oracle_route: {rc}")
    return ids, w


def hist_perm(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    n = T * k
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(n, np.int32)
    inv = np.zeros(n, np.int32)
    rc = lib().oracle_hist_perm(_p(ids), T, k, E, _p(counts), _p(offsets), _p(perm), _p(inv))
    if rc != OK:
        raise ValueError(f"oracle_hist_perm: {rc}")
    return counts, offsets, perm, inv


class LRUPool:
    """One layer's slot pool, stepped one fused (layer, step) event at a time."""

    def __init__(self, slots: int, experts: int, preload: bool = False):
        self.S, self.E = slots, experts
        self.slot_expert = np.full(slots, -1, np.int32)
        self.expert_slot = np.full(experts, -1, np.int32)
        self.stamp = np.zeros(slots, np.int64)
        self.clock = C.c_int64(0)
        self.hits = C.c_int64(0)
        self.misses = C.c_int64(0)
        self.evictions = C.c_int64(0)
        if preload:
            for s in range(min(slots, experts)):
                self.slot_expert[s] = s
                self.expert_slot[s] = s

    def step(self, counts: np.ndarray):
        """Apply one event; returns the list of (expert, slot) loads."""
        counts = _c(counts, np.int32)
        le = np.zeros(self.S, np.int32)
        ls = np.zeros(self.S, np.int32)
        n = np.zeros(1, np.int32)
        rc = lib().oracle_lru_step(self.S, self.E, _p(counts), _p(self.slot_expert), _p(self.expert_slot),
                                   _p(self.stamp), C.byref(self.clock), C.byref(self.hits),
                                   C.byref(self.misses), C.byref(self.evictions), _p(le), _p(ls), _p(n))
        if rc == ERR_CAPACITY:
            raise OverflowError("unique routed experts exceed the slots")
        return list(zip(le[: n[0]].tolist(), ls[: n[0]].tolist()))

    def slot_map(self) -> np.ndarray:
        return self.expert_slot.copy()

    def counters(self) -> dict:
        return dict(hits=self.hits.value, misses=self.misses.value, evictions=self.evictions.value)


# ---- expert FFN --------------------------------------------------------------

def expert_gateup(wt: dict, xf: np.ndarray):
    """One expert's gate/up/SwiGLU on an fp32 input vector -> (g, u, h bf16 bits)."""
    I, H = wt["gate_codes"].shape[0], wt["gate_codes"].shape[1] * 2
    xf = _c(xf, np.float32)
    g = np.zeros(I, np.float32)
    u = np.zeros(I, np.float32)
    h = np.zeros(I, np.uint16)
    lib().oracle_expert_gateup(_p(_c(wt["gate_codes"], np.uint8)), _p(_c(wt["gate_scales"], np.uint8)),
                               _p(_c(wt["up_codes"], np.uint8)), _p(_c(wt["up_scales"], np.uint8)),
                               H, I, _p(xf), _p(g), _p(u), _p(h))
    return g, u, h


def expert_down(wt: dict, hf: np.ndarray) -> np.ndarray:
    H, I = wt["down_codes"].shape[0], wt["down_codes"].shape[1] * 2
    hf = _c(hf, np.float32)
    y = np.zeros(H, np.float32)
    lib().oracle_expert_down(_p(_c(wt["down_codes"], np.uint8)), _p(_c(wt["down_scales"], np.uint8)),
                             H, I, _p(hf), _p(y))
    return y


def layer(x_bf16: np.ndarray, ids: np.ndarray, w: np.ndarray, weights: dict, prefill: bool,
          threads: int = 1, want_intermediates: bool = False):
    """The whole layer.  ``weights`` holds stacked ``[E, ...]`` canonical arrays
    indexed by ``ids``.  Returns ``out`` (fp32 ``[T, H]``), plus a dict of
    intermediates when asked."""
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, H = x.shape
    k = ids.shape[1]
    I = weights["gate_codes"].shape[1]
    out = np.zeros((T, H), np.float32)
    A = T * k
    h = np.zeros((A, I), np.uint16)
    xq = np.zeros((T, H), np.uint8) if (prefill and want_intermediates) else None
    xs = np.zeros((T, H // 32), np.uint8) if (prefill and want_intermediates) else None
    hq = np.zeros((A, I), np.uint8) if (prefill and want_intermediates) else None
    hs = np.zeros((A, I // 32), np.uint8) if (prefill and want_intermediates) else None
    ws = {kk: _c(v, np.uint8) for kk, v in weights.items()}
    rc = lib().oracle_layer(int(bool(prefill)), T, H, I, k, _p(x), _p(ids), _p(w),
                            _p(ws["gate_codes"]), _p(ws["gate_scales"]), _p(ws["up_codes"]),
                            _p(ws["up_scales"]), _p(ws["down_codes"]), _p(ws["down_scales"]),
                            _p(out), _p(h), _p(xq), _p(xs), _p(hq), _p(hs), int(threads))
    if rc != OK:
        raise ValueError(f"oracle_layer: {rc}")
    if want_intermediates:
        return out, dict(h=h, xq=xq, xs=xs, hq=hq, hs=hs)
    return out


def combine(y: np.ndarray, w: np.ndarray) -> np.ndarray:
    y = _c(y, np.float32)
    w = _c(w, np.float32)
    T, k = w.shape
    H = y.shape[-1]
    out = np.zeros((T, H), np.float32)
    lib().oracle_combine(_p(y), _p(w), T, k, H, _p(out))
    return out
