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
  * e2m1_encode / mxfp4_quant_row ..... pinned (hand-worked OCP rounding cases,
                                        brute-force nearest-with-ties-to-even,
                                        scale closed form, dequantised bound)
  * route (top-k + softmax) ........... pinned (brute-force sort, closed forms)
  * hist_perm ......................... pinned (numpy stable argsort, invariants)
  * lru_step .......................... pinned (independent list simulator, hand cases)
  * PolicyPool (lru/fifo/lfu/lfru/slru)  pinned (hand-worked event streams per policy,
                                        LRU mode against lru_step, exhaustive
                                        offline-optimal lower bound on tiny streams)
  * PolicyPool.staged_prefill ......... pinned (hand-worked windows, a case where
                                        keeping the window in flight changes the
                                        LFU victim, load-once and residency
                                        invariants)
  * expert_gateup / expert_down ....... pinned (integer-exact case, float64 numpy bound)
  * layer (decode, prefill, FP4 act) .. pinned piecewise and against a float64
                                        numpy evaluation (brute-force E2M1
                                        nearest for the FP4-activation mode);
                                        the end-to-end float value has no
                                        printed worked example
  * combine ........................... pinned (k=1 identity, float64 bound)
  * f16 / GGUF Q8_0, Q4_K dequant ...... pinned (binary16 against torch over all
                                        codes; hand-worked blocks; structural
                                        special cases of the Q4_K scale/min
                                        packing and nibble order)
  * layer_gguf (decode) ............... pinned against a float64 numpy evaluation
                                        within the fp32 summation bound, and
                                        equal to the MXFP4 layer on weights
                                        both formats represent exactly
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
            L.oracle_e2m1_encode.restype = C.c_uint8
            L.oracle_e2m1_encode.argtypes = [C.c_double]
            L.oracle_mxfp4_quant_row.argtypes = [vp, i32, vp, vp]
            L.oracle_dequant_mxfp4.argtypes = [vp, vp, i32, i32, vp]
            L.oracle_route.argtypes = [vp, i32, i32, i32, vp, vp]
            L.oracle_hist_perm.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
            L.oracle_lru_step.argtypes = [i32, i32, vp, vp, vp, vp, i64p, i64p, i64p, i64p, vp, vp, vp]
            L.oracle_expert_gateup.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp]
            L.oracle_expert_down.argtypes = [vp, vp, i32, i32, vp, vp]
            L.oracle_layer.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                       vp, vp, vp, vp, vp, vp, i32]
            L.oracle_combine.argtypes = [vp, vp, i32, i32, i32, vp]
            L.oracle_f16_value.restype = C.c_double
            L.oracle_f16_value.argtypes = [C.c_uint16]
            L.oracle_dequant_q8_0.argtypes = [vp, i32, i32, vp]
            L.oracle_dequant_q4_k.argtypes = [vp, i32, i32, vp]
            L.oracle_gguf_row_bytes.restype = C.c_long
            L.oracle_gguf_row_bytes.argtypes = [i32, i32]
            L.oracle_layer_gguf.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32]
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


def e2m1_encode(v: float) -> int:
    return lib().oracle_e2m1_encode(v)


def mxfp4_quant(x_bf16_bits: np.ndarray):
    """MXFP4 of each row of ``[rows, K]`` bf16 bits -> (packed codes u8
    ``[rows, K/2]``, scales u8 ``[rows, K/32]``)."""
    x = _c(x_bf16_bits, np.uint16)
    rows, K = x.shape
    q = np.zeros((rows, K // 2), np.uint8)
    s = np.zeros((rows, K // 32), np.uint8)
    for r in range(rows):
        lib().oracle_mxfp4_quant_row(_p(x[r]), K, _p(q[r]), _p(s[r]))
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


POLICIES = ("lru", "fifo", "lfu", "lfru", "slru")


class PolicyPool:
    """One layer's slot pool under any of the named cache policies, written
    out plainly in Python (events are small: E <= 256 experts).

    The policies are named in the tinyserve README ("Configuration":
    cache_policy lru, lfru, slru, lfu, fifo; "How it works" item 3:
    frequency-recency eviction); the pages do not define them, so the
    plainest readings are taken.  One fused event per (layer, step), as the
    replay-semantics study on the Expert Offloading topic page prescribes:
    U = experts with a nonzero count.  First every resident member of U, in
    ascending id, is "routed again"; then every absent member, in ascending
    id, takes the lowest-numbered free slot, or else the slot of a resident
    expert outside U chosen by the policy:
      lru   the one routed longest ago (loading counts as routing)
      fifo  the one loaded longest ago (being routed again does not count)
      lfu   the one routed in the fewest events since it was loaded, then
            the lowest expert id
      lfru  the one routed in the fewest events since it was loaded, then
            the one routed longest ago
      slru  experts are probationary when loaded; routed again, a
            probationary expert becomes protected; when more than
            max(1, S // 2) are protected, the protected one routed longest
            ago becomes probationary again (and counts as just routed);
            the victim is the probationary one routed longest ago, else the
            protected one routed longest ago
    """

    def __init__(self, slots: int, experts: int, policy: str = "lru", preload: bool = False):
        assert policy in POLICIES
        self.S, self.E, self.policy = slots, experts, policy
        self.slot_of = {}          # expert -> slot
        self.last_routed = {}      # expert -> time of last routing (or load)
        self.loaded_at = {}        # expert -> time of load
        self.uses = {}             # expert -> events routed since load (load = 1)
        self.protected = set()     # slru
        self.freq = [0] * experts  # events that routed the expert (prefetch ranking)
        self.fresh = set()         # loaded by a prefetch, not routed since
        self.time = 0
        self.hits = self.misses = self.evictions = 0
        self.prefetches = self.prefetch_hits = 0
        if preload:
            for e in range(min(slots, experts)):
                self._load(e, e)

    def _tick(self):
        self.time += 1
        return self.time

    def _load(self, e, slot):
        self.slot_of[e] = slot
        t = self._tick()
        self.last_routed[e] = t
        self.loaded_at[e] = t
        self.uses[e] = 1
        self.protected.discard(e)

    def _route_again(self, e):
        if self.policy == "fifo":
            return
        if self.policy == "lfu":
            self.uses[e] += 1
            return
        if self.policy == "lfru":
            self.uses[e] += 1
        self.last_routed[e] = self._tick()
        if self.policy == "slru" and e not in self.protected:
            self.protected.add(e)
            if len(self.protected) > max(1, self.S // 2):
                oldest = min(self.protected, key=lambda x: self.last_routed[x])
                self.protected.discard(oldest)
                self.last_routed[oldest] = self._tick()

    def _victim(self, routed):
        cand = [e for e in self.slot_of if e not in routed]
        if self.policy == "fifo":
            return min(cand, key=lambda e: self.loaded_at[e])
        if self.policy == "lfu":
            return min(cand, key=lambda e: (self.uses[e], e))
        if self.policy == "lfru":
            return min(cand, key=lambda e: (self.uses[e], self.last_routed[e]))
        if self.policy == "slru":
            return min(cand, key=lambda e: (e in self.protected, self.last_routed[e]))
        return min(cand, key=lambda e: self.last_routed[e])

    def step(self, counts, keep=()):
        """Apply one event; returns the list of (expert, slot) loads.  Experts
        in ``keep`` (still read by work in flight) are never victims."""
        routed = [e for e in range(self.E) if counts[e] > 0]
        if len(routed) > self.S:
            raise OverflowError("unique routed experts exceed the slots")
        for e in routed:
            if e in self.slot_of:
                self.hits += 1
                if e in self.fresh:
                    self.prefetch_hits += 1
                    self.fresh.discard(e)
                self._route_again(e)
        loads = []
        for e in routed:
            if e in self.slot_of:
                continue
            used = set(self.slot_of.values())
            free = [s for s in range(self.S) if s not in used]
            if free:
                slot = free[0]
            else:
                v = self._victim(set(routed) | set(keep))
                slot = self.slot_of.pop(v)
                self.protected.discard(v)
                self.fresh.discard(v)
                self.evictions += 1
            self._load(e, slot)
            self.misses += 1
            loads.append((e, slot))
        for e in routed:
            self.freq[e] += 1
        return loads

    def prefetch(self, max_loads):
        """Speculative loads ahead of the layer's routing (next-layer
        prefetch; FATE is the pages' example of the idea, driven there by
        the next layer's gate, which this path does not have).  Reading:
        the non-resident experts routed in at least one earlier event, most
        often routed first (ties: lower id), are loaded one by one, at most
        ``max_loads``: into the lowest free slot, else into the policy's
        victim (never one loaded by this call) if that victim was routed in
        fewer events than the candidate; the first candidate without such a
        slot ends the call.  Returns the (expert, slot) loads."""
        cand = sorted((e for e in range(self.E) if e not in self.slot_of and self.freq[e] > 0),
                      key=lambda e: (-self.freq[e], e))
        loads, mine = [], set()
        for e in cand:
            if len(loads) >= max_loads:
                break
            used = set(self.slot_of.values())
            free = [s for s in range(self.S) if s not in used]
            if free:
                slot = free[0]
            else:
                if len(mine) >= len(self.slot_of):
                    break
                v = self._victim(mine)
                if self.freq[v] >= self.freq[e]:
                    break
                slot = self.slot_of.pop(v)
                self.protected.discard(v)
                self.fresh.discard(v)
                self.evictions += 1
            self._load(e, slot)
            self.fresh.add(e)
            mine.add(e)
            self.prefetches += 1
            loads.append((e, slot))
        return loads

    def staged_prefill(self, counts, window):
        """The staging events of one prefill call through a pool smaller than
        the routed set: the routed experts, ascending, cut into windows of at
        most ``window``; each window is one event, and the previous window's
        experts (whose GEMMs may still run) are never its victims.  Returns
        [(window experts, loads)].  Every routed expert sits in exactly one
        window, so none is loaded twice in a call (the pages' "each unique
        expert loaded once" for prefill)."""
        routed = [e for e in range(self.E) if counts[e] > 0]
        out, prev = [], []
        for i in range(0, len(routed), window):
            win = routed[i:i + window]
            cw = [counts[e] if e in win else 0 for e in range(self.E)]
            out.append((win, self.step(cw, keep=prev)))
            prev = win
        return out

    def slot_map(self) -> np.ndarray:
        m = np.full(self.E, -1, np.int32)
        for e, s in self.slot_of.items():
            m[e] = s
        return m

    def counters(self) -> dict:
        return dict(hits=self.hits, misses=self.misses, evictions=self.evictions)

    def prefetch_counters(self) -> dict:
        return dict(prefetches=self.prefetches, prefetch_hits=self.prefetch_hits)


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


_ACT_MODES = {"bf16": 0, "mxfp8": 1, "mxfp4": 2}


def layer(x_bf16: np.ndarray, ids: np.ndarray, w: np.ndarray, weights: dict, prefill: bool,
          threads: int = 1, want_intermediates: bool = False, act: str | None = None):
    """The whole layer.  ``weights`` holds stacked ``[E, ...]`` canonical arrays
    indexed by ``ids``.  Returns ``out`` (fp32 ``[T, H]``), plus a dict of
    intermediates when asked.

    ``act`` picks the expert-input format at both quantisation points (x
    before gate/up, h before down): ``"bf16"`` (the decode path),
    ``"mxfp8"`` (the prefill path) or ``"mxfp4"`` (the FP4-activation
    prefill variant); by default it follows ``prefill``.  With ``"mxfp4"``
    the intermediates ``xq``/``hq`` are packed two codes per byte."""
    if act is None:
        act = "mxfp8" if prefill else "bf16"
    if act not in _ACT_MODES:
        raise ValueError(f"act must be one of {sorted(_ACT_MODES)}, got {act!r}")
    mode = _ACT_MODES[act]
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, H = x.shape
    k = ids.shape[1]
    I = weights["gate_codes"].shape[1]
    out = np.zeros((T, H), np.float32)
    A = T * k
    h = np.zeros((A, I), np.uint16)
    per = 2 if mode == 2 else 1           # elements per code byte
    keep = bool(mode) and want_intermediates
    xq = np.zeros((T, H // per), np.uint8) if keep else None
    xs = np.zeros((T, H // 32), np.uint8) if keep else None
    hq = np.zeros((A, I // per), np.uint8) if keep else None
    hs = np.zeros((A, I // 32), np.uint8) if keep else None
    ws = {kk: _c(v, np.uint8) for kk, v in weights.items()}
    rc = lib().oracle_layer(mode, T, H, I, k, _p(x), _p(ids), _p(w),
                            _p(ws["gate_codes"]), _p(ws["gate_scales"]), _p(ws["up_codes"]),
                            _p(ws["up_scales"]), _p(ws["down_codes"]), _p(ws["down_scales"]),
                            _p(out), _p(h), _p(xq), _p(xs), _p(hq), _p(hs), int(threads))
    if rc != OK:
        raise ValueError(f"oracle_layer: {rc}")
    if want_intermediates:
        return out, dict(h=h, xq=xq, xs=xs, hq=hq, hs=hs)
    return out


GGUF_FORMATS = {"q8_0": 0, "q4_k": 1}


def f16_value(bits: int) -> float:
    """IEEE binary16 bit pattern -> value (from the bit definition)."""
    return lib().oracle_f16_value(int(bits))


def gguf_row_bytes(fmt: str, K: int) -> int:
    """Bytes of one row of ``K`` elements in GGUF ``fmt`` (0 if K does not fit)."""
    return int(lib().oracle_gguf_row_bytes(GGUF_FORMATS[fmt], int(K)))


def dequant_gguf(fmt: str, blocks: np.ndarray, K: int) -> np.ndarray:
    """Rows of GGUF blocks ``[rows, row_bytes]`` (``"q8_0"`` or ``"q4_k"``)
    -> fp32 ``[rows, K]``, by the format's rule (moe_oracle.c)."""
    rb = gguf_row_bytes(fmt, K)
    if not rb:
        raise ValueError(f"K={K} does not fit {fmt}")
    b = _c(blocks, np.uint8).reshape(-1, rb)
    out = np.zeros((b.shape[0], K), np.float32)
    fn = lib().oracle_dequant_q8_0 if fmt == "q8_0" else lib().oracle_dequant_q4_k
    fn(_p(b), b.shape[0], int(K), _p(out))
    return out


def layer_gguf(fmt: str, x_bf16: np.ndarray, ids: np.ndarray, w: np.ndarray, weights: dict,
               threads: int = 1, want_h: bool = False):
    """The decode layer on GGUF expert weights.  ``weights`` holds stacked
    ``gate``/``up`` ``[E, I, row_bytes(H)]`` and ``down`` ``[E, H,
    row_bytes(I)]`` block bytes.  Returns ``out`` (fp32 ``[T, H]``), and the
    bf16 bits of h ``[T*k, I]`` when asked."""
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, H = x.shape
    k = ids.shape[1]
    g = _c(weights["gate"], np.uint8)
    u = _c(weights["up"], np.uint8)
    d = _c(weights["down"], np.uint8)
    E, I = g.shape[0], g.shape[1]
    if g.shape[2] != gguf_row_bytes(fmt, H) or d.shape[1:] != (H, gguf_row_bytes(fmt, I)) or u.shape != g.shape:
        raise ValueError("weight shapes do not match the format")
    out = np.zeros((T, H), np.float32)
    h = np.zeros((T * k, I), np.uint16)
    rc = lib().oracle_layer_gguf(GGUF_FORMATS[fmt], T, H, I, k, _p(x), _p(ids), _p(w), _p(g), _p(u), _p(d),
                                 E, _p(out), _p(h), int(threads))
    if rc != OK:
        raise ValueError(f"oracle_layer_gguf: {rc}")
    return (out, h) if want_h else out


def combine(y: np.ndarray, w: np.ndarray) -> np.ndarray:
    y = _c(y, np.float32)
    w = _c(w, np.float32)
    T, k = w.shape
    H = y.shape[-1]
    out = np.zeros((T, H), np.float32)
    lib().oracle_combine(_p(y), _p(w), T, k, H, _p(out))
    return out
