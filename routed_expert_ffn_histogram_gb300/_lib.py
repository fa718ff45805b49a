"""ctypes binding of ``libmoe_gb300.so`` (declared in ``include/moe.h``).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  Tensors are passed as raw pointers (``tensor.data_ptr()``),
streams as ``cudaStream_t`` handles.  If the library is not built, every
call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID = -1
MOE_ERR_CUDA = -2
MOE_ERR_CAPACITY = -3
MOE_ERR_TIMEOUT = -4
MOE_ERR_STATE = -5
MOE_ERR_UNSUPPORTED = -6
MOE_MAX_EXPERTS = 256
MOE_MAX_TOPK = 32
MOE_PATH_AUTO = 0
MOE_PATH_DECODE = 1
MOE_PATH_PREFILL = 2
MOE_DECODE_MAX_ASSIGN = 64
MOE_FFN_ACCUMULATE = 0x100
MOE_FFN_SKIP_ABSENT = 0x200
MOE_POLICY_LRU, MOE_POLICY_FIFO, MOE_POLICY_LFU, MOE_POLICY_LFRU, MOE_POLICY_SLRU = 0, 1, 2, 3, 4
POLICIES = {"lru": 0, "fifo": 1, "lfu": 2, "lfru": 3, "slru": 4}
MOE_STAGE_WHOLE, MOE_STAGE_DECODE = 0, 1
MOE_GGUF_Q8_0, MOE_GGUF_Q4_K = 0, 1
GGUF_FORMATS = {"q8_0": MOE_GGUF_Q8_0, "q4_k": MOE_GGUF_Q4_K}

# Every symbol the header declares, with (restype, argtypes).
_vp, _i32, _sz = C.c_void_p, C.c_int, C.c_size_t
_szp = C.POINTER(C.c_size_t)


class MoePoolDesc(C.Structure):
    _fields_ = [("layers", C.c_int), ("experts", C.c_int), ("slots_per_layer", C.c_int),
                ("hidden", C.c_int), ("inter", C.c_int), ("host_experts", C.c_void_p),
                ("dev_slots", C.c_void_p), ("preload", C.c_int), ("dry_run", C.c_int), ("policy", C.c_int),
                ("stage_parts", C.c_int)]


class MoeCounters(C.Structure):
    _fields_ = [("hits", C.c_uint64), ("misses", C.c_uint64), ("evictions", C.c_uint64),
                ("h2d_bytes", C.c_uint64), ("errors", C.c_uint64), ("events", C.c_uint64),
                ("prefetches", C.c_uint64), ("prefetch_hits", C.c_uint64)]

    def as_dict(self):
        return {f: int(getattr(self, f)) for f, _ in self._fields_}


SIGNATURES = {
    "moe_status_str": (C.c_char_p, [_i32]),
    "moe_last_cuda_error": (_i32, []),
    "moe_device_count": (_i32, []),
    "moe_expert_bytes": (_i32, [_i32, _i32, _szp]),
    "moe_pack_expert": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp]),
    "moe_route_workspace_bytes": (_i32, [_i32, _i32, _i32, _szp]),
    "moe_route_plan": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_route_plan_noalloc": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_pool_create": (_i32, [C.POINTER(MoePoolDesc), C.POINTER(C.c_void_p)]),
    "moe_pool_stage": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp, _i32]),
    "moe_prefill_staged": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _sz, _vp,
                                  _vp, _vp, _i32]),
    "moe_pool_prefetch": (_i32, [_vp, _i32, _i32, _vp, _vp, C.POINTER(C.c_int)]),
    "moe_pool_counters": (_i32, [_vp, _i32, C.POINTER(MoeCounters)]),
    "moe_pool_slot_map": (_i32, [_vp, _i32, _vp]),
    "moe_pool_last_loads": (_i32, [_vp, _i32, _vp, _vp, C.POINTER(C.c_int)]),
    "moe_pool_state_bytes": (_i32, [_vp, _szp]),
    "moe_pool_save": (_i32, [_vp, _vp, _sz]),
    "moe_pool_load": (_i32, [_vp, _vp, _sz]),
    "moe_pool_inject_copy_failures": (_i32, [_vp, _i32]),
    "moe_pool_device_state_bytes": (_i32, [_vp, _szp]),
    "moe_pool_device_attach": (_i32, [_vp, _vp, _sz, _vp, _i32]),
    "moe_pool_stage_device": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp]),
    "moe_pool_route_stage_device": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                           _vp]),
    "moe_pool_device_join": (_i32, [_vp, _i32, _vp]),
    "moe_pool_device_detach": (_i32, [_vp, _vp, _i32]),
    "moe_pool_destroy": (None, [_vp]),
    "moe_ffn_workspace_bytes": (_i32, [_i32, _i32, _i32, _i32, _i32, _szp]),
    "moe_expert_ffn": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _sz, _vp,
                              _vp]),
    "moe_decode_layer": (_i32, [_vp, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                                _vp]),
    "moe_decode_layer_acc": (_i32, [_vp, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                    _vp, _vp]),
    "moe_ffn_status": (_i32, [_vp, _i32, _vp, C.POINTER(C.c_uint32)]),
    "moe_debug_stall_next_decode": (_i32, [_i32]),
    "moe_combine": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp]),
    "moe_quant_mxfp4": (_i32, [_vp, _i32, _i32, _vp, _vp, _i32, _vp]),
    "moe_quant_mxfp8": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _i32, _vp]),
    "moe_probe_mxf8f6f4": (_i32, [_i32, _vp, C.POINTER(C.c_int), _vp]),
    "moe_gguf_expert_bytes": (_i32, [_i32, _i32, _i32, _szp]),
    "moe_gguf_workspace_bytes": (_i32, [_i32, _i32, _i32, _i32, _szp]),
    "moe_expert_ffn_gguf": (_i32, [_i32, _vp, _i32, _i32, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _vp, _sz,
                                   _vp, _i32, _vp]),
    "moe_decode_layer_gguf": (_i32, [_i32, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _vp, _i32, _vp, _sz, _vp, _i32, _vp]),
}

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn, status, cuda_err=0):
        self.status = status
        self.cuda_error = cuda_err
        msg = f"{fn}: {status_str(status)} ({status})"
        if status == MOE_ERR_CUDA:
            msg += f", CUDA error {cuda_err}"
        super().__init__(msg)


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library missing: {LIB_PATH}; build it with "
                                   "routed_expert_ffn_histogram_gb300.build.build()")
            L = C.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().moe_status_str(status).decode()


def check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status, lib().moe_last_cuda_error() if status == MOE_ERR_CUDA else 0)
    return status


def ptr(t):
    """Raw address of a tensor / numpy array / int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(type(t))


def stream_handle(stream=None):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
