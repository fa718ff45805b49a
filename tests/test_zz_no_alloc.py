"""moe_route_plan_noalloc: routing for callers that cannot allocate device
memory (engines whose device memory belongs to their own fixed-budget
allocator, decode loops that must stay out of the driver's allocator).  It
keeps its tile histograms in the library's own device array instead of a
caller workspace, so its results must equal moe_route_plan's exactly --
including on a second call, which finds the first call's data still in the
shared array.  Called through the C ABI with raw pointers."""
import numpy as np
import pytest

import moe_synth as S
from helpers import ULP_TOL_W, f32_ulp_diff

pytestmark = pytest.mark.gpu


def _buffers(T, E, k):
    import torch

    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(ids=torch.full((T, k), -1, **i32), w=torch.full((T, k), -1.0, device="cuda"),
                counts=torch.full((E,), -1, **i32), offsets=torch.full((E + 1,), -1, **i32),
                perm=torch.full((T * k,), -1, **i32), inv=torch.full((T * k,), -1, **i32))


def _noalloc(L, lg, k, b, stream):
    T, E = lg.shape
    return L.moe_route_plan_noalloc(lg.data_ptr(), T, E, k, b["ids"].data_ptr(), b["w"].data_ptr(),
                                    b["counts"].data_ptr(), b["offsets"].data_ptr(), b["perm"].data_ptr(),
                                    b["inv"].data_ptr(), None, stream)


def _with_workspace(L, lg, k, b, stream):
    import torch

    T, E = lg.shape
    import ctypes as C

    need = C.c_size_t(0)
    assert L.moe_route_workspace_bytes(T, E, k, C.byref(need)) == 0
    ws = torch.empty(max(need.value, 16), dtype=torch.uint8, device="cuda")
    rc = L.moe_route_plan(lg.data_ptr(), T, E, k, b["ids"].data_ptr(), b["w"].data_ptr(), b["counts"].data_ptr(),
                          b["offsets"].data_ptr(), b["perm"].data_ptr(), b["inv"].data_ptr(), None,
                          ws.data_ptr(), ws.numel(), stream)
    return rc, ws


def test_noalloc_matches_workspace_route_twice():
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    L = M.lib()
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row on the same array: the largest allowed size first
    # (16384 tokens, 128 experts, top-8), then a smaller one
    cases = [(S.WORKLOADS[4], S.logits(S.WORKLOADS[4], 0)), (S.WORKLOADS[3], S.logits(S.WORKLOADS[3], 0))]
    for wl, logits in cases:
        T, E = logits.shape
        lg = torch.from_numpy(logits).cuda()
        a, b = _buffers(T, E, wl.top_k), _buffers(T, E, wl.top_k)
        assert _noalloc(L, lg, wl.top_k, a, stream) == M.MOE_OK
        rc, ws = _with_workspace(L, lg, wl.top_k, b, stream)
        assert rc == M.MOE_OK
        torch.cuda.synchronize()
        for key in ("ids", "counts", "offsets", "perm", "inv"):
            assert torch.equal(a[key], b[key]), key
        assert np.all(f32_ulp_diff(a["w"].cpu().numpy(), b["w"].cpu().numpy()) <= ULP_TOL_W)


def test_noalloc_rejects_sizes_beyond_its_array():
    import routed_expert_ffn_histogram_gb300 as M

    L = M.lib()
    # 16385 tokens need a 65th tile: refused before anything is enqueued
    assert L.moe_route_plan_noalloc(1, 16385, 8, 2, 1, 1, 1, 1, 1, 1, None, None) == M.MOE_ERR_INVALID
