"""Routed-expert FFN over a fixed GPU expert-slot pool, for GB300 (sm_103a).

Python face of the C library declared in ``include/moe.h``.  The functions
keep the C names and only marshal arguments (torch tensors -> pointers,
torch streams -> ``cudaStream_t``); every computation runs in the library's
CUDA kernels.  PyTorch provides device memory, pinned host memory and
streams.

Typical use for one layer and one step::

    plan = RoutePlan.allocate(T, E, k, device)
    moe_route_plan(logits, k, plan)                      # top-k, histogram, perm
    pool.stage(layer, plan.counts_host, slot_of)         # LRU + miss copies
    moe_expert_ffn(pool, layer, x, plan, slot_of, out)   # experts + combine
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

from . import _lib
from ._lib import (MOE_DECODE_MAX_ASSIGN, MOE_FFN_ACCUMULATE, MOE_FFN_SKIP_ABSENT, MOE_ERR_CAPACITY, MOE_ERR_CUDA, MOE_ERR_INVALID, MOE_ERR_STATE,
                   MOE_ERR_TIMEOUT, MOE_ERR_UNSUPPORTED, MOE_MAX_EXPERTS, MOE_MAX_TOPK, MOE_OK,
                   MOE_PATH_AUTO, MOE_PATH_DECODE, MOE_PATH_PREFILL, MOE_POLICY_FIFO, MOE_POLICY_LFRU,
                   MOE_POLICY_LFU, MOE_POLICY_LRU, MOE_POLICY_SLRU, MOE_STAGE_DECODE,
                   MOE_STAGE_WHOLE, POLICIES, GGUF_FORMATS, MOE_GGUF_Q8_0, MOE_GGUF_Q4_K, MoeCounters, MoeError,
                   MoePoolDesc,
                   check,
                   lib, ptr, status_str, stream_handle)

__all__ = [
    "moe_expert_bytes", "moe_pack_expert", "moe_route_workspace_bytes", "moe_route_plan", "moe_route_plan_noalloc",
    "moe_ffn_workspace_bytes", "alloc_ffn_workspace",
    "moe_expert_ffn", "moe_decode_layer", "moe_ffn_status", "moe_debug_stall_next_decode", "moe_combine",
    "moe_quant_mxfp8", "moe_quant_mxfp4", "moe_probe_mxf8f6f4", "moe_gguf_expert_bytes", "pack_gguf_expert",
    "moe_expert_ffn_gguf", "moe_decode_layer_gguf", "alloc_gguf_workspace", "gguf_workspace_h", "GGUF_FORMATS", "Pool", "RoutePlan", "MoeCounters", "MoeError", "lib", "status_str",
    "POLICIES", "MOE_PATH_AUTO", "MOE_PATH_DECODE", "MOE_PATH_PREFILL", "MOE_FFN_ACCUMULATE", "MOE_FFN_SKIP_ABSENT",
]


def moe_expert_bytes(hidden: int, inter: int) -> int:
    out = C.c_size_t(0)
    check("moe_expert_bytes", lib().moe_expert_bytes(hidden, inter, C.byref(out)))
    return out.value


def moe_pack_expert(w: dict, hidden: int, inter: int, dst) -> None:
    """Canonical MXFP4 arrays (host numpy, see ``include/moe.h``) -> native
    layout written at host address/array ``dst``."""
    import numpy as np

    a = {k: np.ascontiguousarray(v, np.uint8) for k, v in w.items()}
    check("moe_pack_expert", lib().moe_pack_expert(
        ptr(a["gate_codes"]), ptr(a["gate_scales"]), ptr(a["up_codes"]), ptr(a["up_scales"]),
        ptr(a["down_codes"]), ptr(a["down_scales"]), hidden, inter, ptr(dst)))


def moe_route_workspace_bytes(T: int, E: int, k: int) -> int:
    out = C.c_size_t(0)
    check("moe_route_workspace_bytes", lib().moe_route_workspace_bytes(T, E, k, C.byref(out)))
    return out.value


@dataclass
class RoutePlan:
    """Device buffers written by moe_route_plan (plus optional pinned counts)."""

    T: int
    E: int
    k: int
    ids: object
    w: object
    counts: object
    offsets: object
    perm: object
    inv: object
    workspace: object
    counts_host: object = None

    @staticmethod
    def allocate(T: int, E: int, k: int, device="cuda", counts_host: bool = False) -> "RoutePlan":
        import torch

        i32 = dict(dtype=torch.int32, device=device)
        ws = max(moe_route_workspace_bytes(T, E, k), 16)
        return RoutePlan(T, E, k,
                         ids=torch.empty((T, k), **i32), w=torch.empty((T, k), dtype=torch.float32, device=device),
                         counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
                         perm=torch.empty(max(T * k, 1), **i32), inv=torch.empty(max(T * k, 1), **i32),
                         workspace=torch.empty(ws, dtype=torch.uint8, device=device),
                         counts_host=torch.empty(E, dtype=torch.int32).pin_memory() if counts_host else None)


def moe_route_plan(logits, k: int, plan: RoutePlan, stream=None, with_counts_host: bool = True) -> None:
    """Top-k + softmax + histogram + stable permutation (moe_route_plan)."""
    T, E = logits.shape
    ch = plan.counts_host if with_counts_host else None
    check("moe_route_plan", lib().moe_route_plan(
        ptr(logits), T, E, k, ptr(plan.ids), ptr(plan.w), ptr(plan.counts), ptr(plan.offsets), ptr(plan.perm),
        ptr(plan.inv), ptr(ch), ptr(plan.workspace), plan.workspace.numel(), stream_handle(stream)))


def moe_route_plan_noalloc(logits, k: int, plan: RoutePlan, stream=None, with_counts_host: bool = True) -> None:
    """moe_route_plan for callers that cannot allocate device memory: the
    library's own device array replaces the workspace (T <= 16384; calls
    that overlap on the GPU race on it).  ``plan.workspace`` is not used."""
    T, E = logits.shape
    ch = plan.counts_host if with_counts_host else None
    check("moe_route_plan_noalloc", lib().moe_route_plan_noalloc(
        ptr(logits), T, E, k, ptr(plan.ids), ptr(plan.w), ptr(plan.counts), ptr(plan.offsets), ptr(plan.perm),
        ptr(plan.inv), ptr(ch), stream_handle(stream)))


def moe_ffn_workspace_bytes(T: int, k: int, hidden: int, inter: int, path: int = MOE_PATH_AUTO) -> int:
    out = C.c_size_t(0)
    check("moe_ffn_workspace_bytes", lib().moe_ffn_workspace_bytes(T, k, hidden, inter, path, C.byref(out)))
    return out.value


def alloc_ffn_workspace(T: int, k: int, hidden: int, inter: int, path: int = MOE_PATH_AUTO, device="cuda"):
    """A zeroed device workspace for moe_expert_ffn / moe_decode_layer (the
    decode path keeps a completion counter and an fp32 accumulator in it
    that must start at zero; the library leaves them zero)."""
    import torch

    n = max(moe_ffn_workspace_bytes(T, k, hidden, inter, path), 256)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_expert_ffn(pool: "Pool", layer: int, x_bf16, plan: RoutePlan, slot_of, out, workspace,
                   path: int = MOE_PATH_AUTO, stream=None, accumulate: bool = False,
                   skip_absent: bool = False) -> None:
    """Routed experts of one layer with the weighted combine (moe_expert_ffn);
    ``accumulate`` adds into ``out`` (a residual stream) instead of
    overwriting it; ``skip_absent`` serves only the assignments whose
    expert's ``slot_of`` entry is >= 0 (decode path)."""
    T = x_bf16.shape[0]
    if accumulate:
        path |= MOE_FFN_ACCUMULATE
    if skip_absent:
        path |= MOE_FFN_SKIP_ABSENT
    check("moe_expert_ffn", lib().moe_expert_ffn(
        pool.handle, layer, ptr(x_bf16), T, plan.k, ptr(plan.ids), ptr(plan.w), ptr(plan.offsets),
        ptr(plan.perm), ptr(plan.inv), ptr(slot_of), path, ptr(workspace),
        workspace.numel() * workspace.element_size() if workspace is not None else 0, ptr(out),
        stream_handle(stream)))


def moe_decode_layer(pool: "Pool", layer: int, logits, x_bf16, plan: RoutePlan, slot_of, out, workspace,
                     stream=None, accumulate: bool = False) -> None:
    """Routing + routed experts of one decode step in one launch
    (moe_decode_layer); fills ``plan`` like moe_route_plan.  ``accumulate``
    adds into ``out`` (moe_decode_layer_acc) instead of overwriting it."""
    T = x_bf16.shape[0]
    fn = lib().moe_decode_layer_acc if accumulate else lib().moe_decode_layer
    check("moe_decode_layer", fn(
        pool.handle, layer, ptr(logits), ptr(x_bf16), T, plan.k, ptr(plan.ids), ptr(plan.w), ptr(plan.counts),
        ptr(plan.offsets), ptr(plan.perm), ptr(plan.inv), ptr(slot_of), ptr(workspace),
        workspace.numel() * workspace.element_size(), ptr(out), stream_handle(stream)))


def moe_ffn_status(workspace, path: int, stream=None) -> int:
    """Status bits of the kernels that used ``workspace`` (0: every bounded
    wait completed); waits for ``stream`` and clears them (moe_ffn_status)."""
    bits = C.c_uint32(0)
    check("moe_ffn_status", lib().moe_ffn_status(ptr(workspace), path, stream_handle(stream), C.byref(bits)))
    return bits.value


def moe_debug_stall_next_decode(n: int = 1) -> None:
    """Test hook: the next n fused decode launches time out on purpose."""
    check("moe_debug_stall_next_decode", lib().moe_debug_stall_next_decode(n))


def moe_combine(y_perm, w, inv, out, stream=None) -> None:
    T, k = w.shape
    H = out.shape[1]
    check("moe_combine", lib().moe_combine(ptr(y_perm), ptr(w), ptr(inv), T, k, H, ptr(out),
                                           stream_handle(stream)))


def moe_quant_mxfp4(x_bf16, q, scales, stream=None) -> None:
    """MXFP4 of bf16 rows: q uint8 [rows][K/2] (two codes per byte), scales
    uint8 [rows][>= K/32] (moe_quant_mxfp4)."""
    rows, K = x_bf16.shape
    check("moe_quant_mxfp4", lib().moe_quant_mxfp4(ptr(x_bf16), K, rows, ptr(q), ptr(scales), scales.shape[1],
                                                   stream_handle(stream)))


def moe_quant_mxfp8(x_bf16, q, scales, perm=None, k: int = 1, stream=None) -> None:
    rows, K = q.shape
    check("moe_quant_mxfp8", lib().moe_quant_mxfp8(ptr(x_bf16), K, ptr(perm), k, rows, ptr(q), ptr(scales),
                                                   scales.shape[1], stream_handle(stream)))


def _fmt(fmt) -> int:
    return GGUF_FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def moe_gguf_expert_bytes(fmt, hidden: int, inter: int) -> int:
    out = C.c_size_t(0)
    check("moe_gguf_expert_bytes", lib().moe_gguf_expert_bytes(_fmt(fmt), hidden, inter, C.byref(out)))
    return out.value


def pack_gguf_expert(w: dict, fmt, hidden: int, inter: int, dst) -> None:
    """One GGUF expert's raw rows (host numpy ``gate``/``up`` [I][row bytes],
    ``down`` [H][row bytes]) placed back to back into its slot image at the
    host address / array ``dst`` (``moe_gguf_expert_bytes`` bytes)."""
    import numpy as np

    eb = moe_gguf_expert_bytes(fmt, hidden, inter)
    parts = [np.ascontiguousarray(w[k], np.uint8).reshape(-1) for k in ("gate", "up", "down")]
    img = np.zeros(eb, np.uint8)
    o = 0
    for part in parts:
        img[o:o + part.size] = part
        o += part.size
    if o > eb:
        raise ValueError("weight shapes do not match the format")
    C.memmove(ptr(dst), img.ctypes.data, eb)


def alloc_gguf_workspace(T: int, k: int, hidden: int, inter: int, device="cuda"):
    import torch

    out = C.c_size_t(0)
    check("moe_gguf_workspace_bytes", lib().moe_gguf_workspace_bytes(T, k, hidden, inter, C.byref(out)))
    # zero-filled: the single-launch kernel keeps its cross-CTA counters here
    return torch.zeros(max(out.value, 256), dtype=torch.uint8, device=device)


def gguf_workspace_h(workspace, T: int, k: int, inter: int):
    """The bf16 h [T*k][inter] held in a GGUF workspace (from byte 256), as
    uint16 bits."""
    import torch

    return workspace[256:256 + T * k * inter * 2].view(torch.int16).view(T * k, inter)


def moe_expert_ffn_gguf(fmt, slots, n_slots: int, hidden: int, inter: int, x_bf16, plan: "RoutePlan", slot_of,
                        n_experts: int, out, workspace, accumulate: bool = False, stream=None) -> None:
    """The routed experts on GGUF weights (``moe_expert_ffn_gguf``); ``plan``
    holds ids and w from ``moe_route_plan``."""
    T = x_bf16.shape[0]
    k = plan.ids.shape[1]
    check("moe_expert_ffn_gguf",
          lib().moe_expert_ffn_gguf(_fmt(fmt), ptr(slots), n_slots, hidden, inter, ptr(x_bf16), T, k,
                                    ptr(plan.ids), ptr(plan.w), ptr(slot_of), n_experts, ptr(workspace),
                                    workspace.numel(), ptr(out), 1 if accumulate else 0, stream_handle(stream)))


def moe_decode_layer_gguf(fmt, slots, n_slots: int, hidden: int, inter: int, logits, x_bf16, plan: "RoutePlan",
                          slot_of, n_experts: int, out, workspace, accumulate: bool = False, stream=None) -> None:
    """Routing + routed GGUF experts of one decode step in one launch
    (``moe_decode_layer_gguf``); fills ``plan`` like moe_route_plan."""
    T = x_bf16.shape[0]
    check("moe_decode_layer_gguf", lib().moe_decode_layer_gguf(
        _fmt(fmt), ptr(slots), n_slots, hidden, inter, ptr(logits), ptr(x_bf16), T, plan.k, ptr(plan.ids),
        ptr(plan.w), ptr(plan.counts), ptr(plan.offsets), ptr(plan.perm), ptr(plan.inv), ptr(slot_of), n_experts,
        ptr(workspace), workspace.numel(), ptr(out), 1 if accumulate else 0, stream_handle(stream)))


def moe_probe_mxf8f6f4(stages: int, status, stream=None) -> int:
    """Launch the tensor-core rate probe; returns the CTAs launched.  FLOPs
    per launch: ctas * stages * 4 * 2 * 128 * 256 * 32.  ``status``: a zeroed
    device int32 tensor of one element (bit 1: the completion wait ran out)."""
    n = C.c_int(0)
    check("moe_probe_mxf8f6f4", lib().moe_probe_mxf8f6f4(stages, ptr(status), C.byref(n), stream_handle(stream)))
    return n.value


class Pool:
    """An expert-slot pool (moe_pool_*).  Buffers stay owned by the caller
    (kept referenced here so they outlive the pool)."""

    def __init__(self, layers, experts, slots, hidden, inter, host_experts=None, dev_slots=None,
                 preload=False, dry_run=False, policy=0, stage_parts=0):
        self.layers, self.experts, self.slots, self.hidden, self.inter = layers, experts, slots, hidden, inter
        self.dry_run = bool(dry_run)
        self._keep = (host_experts, dev_slots)
        if isinstance(policy, str):
            policy = POLICIES[policy]
        d = MoePoolDesc(layers, experts, slots, hidden, inter, ptr(host_experts), ptr(dev_slots),
                        int(bool(preload)), int(bool(dry_run)), int(policy),
                        {"whole": 0, "decode": 1}.get(stage_parts, stage_parts))
        h = C.c_void_p()
        check("moe_pool_create", lib().moe_pool_create(C.byref(d), C.byref(h)))
        self.handle = h.value

    def stage(self, layer, counts_host, slot_of_dev=None, compute=None, copy=None, timeout_ms=10000) -> int:
        """One fused cache event; returns the status (raises on errors other
        than capacity and timeout, which are returned)."""
        comp = stream_handle(compute) if (compute is not None or slot_of_dev is not None) else None
        cop = stream_handle(copy) if copy is not None else comp
        rc = lib().moe_pool_stage(self.handle, layer, ptr(counts_host), ptr(slot_of_dev), comp, cop, timeout_ms)
        if rc in (MOE_OK, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT):
            return rc
        check("moe_pool_stage", rc)
        return rc

    def prefill_staged(self, layer, counts_host, window, k, x_bf16=None, plan: RoutePlan = None, out=None,
                       workspace=None, compute=None, copy=None, timeout_ms=10000, T=None) -> None:
        """Prefill of one layer through this pool in windows of at most
        ``window`` unique experts (moe_prefill_staged).  ``counts_host`` is
        the routing's pinned per-expert counts.  On a dry-run pool only the
        staging bookkeeping runs: pass T and leave the tensors out."""
        if T is None:
            T = x_bf16.shape[0]
        comp = None if self.dry_run else stream_handle(compute)
        cop = None if self.dry_run else (stream_handle(copy) if copy is not None else comp)
        p = plan
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        check("moe_prefill_staged", lib().moe_prefill_staged(
            self.handle, layer, ptr(x_bf16), T, k, ptr(p.ids) if p else None, ptr(p.w) if p else None,
            ptr(p.offsets) if p else None, ptr(p.perm) if p else None, ptr(p.inv) if p else None,
            ptr(counts_host), window, ptr(workspace), ws_bytes, ptr(out), comp, cop, timeout_ms))

    def prefetch(self, layer, max_loads, compute=None, copy=None) -> int:
        """Speculative staging of ``layer`` ahead of its routing
        (moe_pool_prefetch); returns the number of experts copied in."""
        comp = None if self.dry_run else stream_handle(compute)
        cop = None if self.dry_run else (stream_handle(copy) if copy is not None else comp)
        n = C.c_int(0)
        check("moe_pool_prefetch", lib().moe_pool_prefetch(self.handle, layer, max_loads, comp, cop, C.byref(n)))
        return n.value

    def device_state_bytes(self) -> int:
        """Bytes of the device buffer that device-planned staging keeps the
        pool's state in (moe_pool_device_state_bytes)."""
        n = C.c_size_t(0)
        check("moe_pool_device_state_bytes", lib().moe_pool_device_state_bytes(self.handle, C.byref(n)))
        return n.value

    def device_attach(self, dev_state, stream=None, timeout_ms=10000) -> None:
        """Move the pool's state into ``dev_state`` (a device tensor of at
        least device_state_bytes() bytes) for device-planned staging."""
        nbytes = dev_state.numel() * dev_state.element_size()
        check("moe_pool_device_attach", lib().moe_pool_device_attach(
            self.handle, ptr(dev_state), nbytes, stream_handle(stream), timeout_ms))

    def stage_device(self, layer, counts_dev, slot_of_dev, split_dev=None, stream=None, copy=None) -> None:
        """Enqueue one staging event planned on the GPU from the device
        counts: slot map into ``slot_of_dev`` (and, with ``split_dev``, the
        hits' and the loads' maps), misses copied by the SMs from the mapped
        host store on ``copy`` (or ``stream``) (moe_pool_stage_device)."""
        check("moe_pool_stage_device", lib().moe_pool_stage_device(
            self.handle, layer, ptr(counts_dev), ptr(slot_of_dev), ptr(split_dev), stream_handle(stream),
            stream_handle(copy) if copy is not None else None))

    def route_stage_device(self, layer, logits, k, plan, slot_of_dev, split_dev=None, stream=None,
                           copy=None) -> None:
        """Route ``logits`` (device fp32 [T, E], T * k <= 32) into ``plan``
        and plan the layer's staging event from the routing in the same
        launch; maps and copies as stage_device (moe_pool_route_stage_device)."""
        T = int(logits.shape[0])
        check("moe_pool_route_stage_device", lib().moe_pool_route_stage_device(
            self.handle, layer, ptr(logits), T, k, ptr(plan.ids), ptr(plan.w), ptr(plan.counts), ptr(plan.offsets),
            ptr(plan.perm), ptr(plan.inv), ptr(slot_of_dev), ptr(split_dev), stream_handle(stream),
            stream_handle(copy) if copy is not None else None))

    def device_join(self, layer, stream=None) -> None:
        """``stream`` waits for the layer's copies on the copy stream
        (moe_pool_device_join)."""
        check("moe_pool_device_join", lib().moe_pool_device_join(self.handle, layer, stream_handle(stream)))

    def device_detach(self, stream=None, timeout_ms=10000) -> int:
        """Bring the state back from the device; returns the status
        (MOE_ERR_CAPACITY or MOE_ERR_INVALID report an event that changed
        nothing; other errors raise)."""
        rc = lib().moe_pool_device_detach(self.handle, stream_handle(stream), timeout_ms)
        if rc in (MOE_OK, MOE_ERR_CAPACITY, MOE_ERR_INVALID):
            return rc
        check("moe_pool_device_detach", rc)
        return rc

    def counters(self, layer=-1) -> dict:
        c = MoeCounters()
        check("moe_pool_counters", lib().moe_pool_counters(self.handle, layer, C.byref(c)))
        return c.as_dict()

    def slot_map(self, layer):
        import numpy as np

        m = np.zeros(self.experts, np.int32)
        check("moe_pool_slot_map", lib().moe_pool_slot_map(self.handle, layer, m.ctypes.data))
        return m

    def last_loads(self, layer):
        import numpy as np

        le = np.zeros(self.slots, np.int32)
        ls = np.zeros(self.slots, np.int32)
        n = C.c_int(0)
        check("moe_pool_last_loads", lib().moe_pool_last_loads(self.handle, layer, le.ctypes.data,
                                                                ls.ctypes.data, C.byref(n)))
        return list(zip(le[: n.value].tolist(), ls[: n.value].tolist()))

    def save(self) -> bytes:
        n = C.c_size_t(0)
        check("moe_pool_state_bytes", lib().moe_pool_state_bytes(self.handle, C.byref(n)))
        buf = C.create_string_buffer(n.value)
        check("moe_pool_save", lib().moe_pool_save(self.handle, buf, n.value))
        return buf.raw

    def load(self, state: bytes) -> int:
        buf = C.create_string_buffer(state, len(state))
        return lib().moe_pool_load(self.handle, buf, len(state))

    def inject_copy_failures(self, n: int) -> None:
        check("moe_pool_inject_copy_failures", lib().moe_pool_inject_copy_failures(self.handle, n))

    def close(self):
        if getattr(self, "handle", None):
            lib().moe_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
