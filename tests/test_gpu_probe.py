"""The tensor-core rate probe behind the prefill roofline: it runs to
completion (its bounded wait reports nothing), its rate scales with the
work asked for, and the rate lies between the published bf16 dense rate and
twice the published FP8 dense rate of the part."""
import pytest

pytestmark = pytest.mark.gpu


def _rate(M, torch, stages, status):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    ctas = M.moe_probe_mxf8f6f4(stages, status)
    b.record()
    torch.cuda.synchronize()
    return ctas * stages * 4 * 2.0 * 128 * 256 * 32 / (a.elapsed_time(b) / 1e3) / 1e12, a.elapsed_time(b)


def test_probe_rate_and_status():
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_probe_mxf8f6f4(64, status)  # warm-up
    torch.cuda.synchronize()
    r1, t1 = _rate(M, torch, 1024, status)
    r2, t2 = _rate(M, torch, 4096, status)
    assert int(status.item()) == 0
    assert t2 > 2.0 * t1                    # time grows with the stages issued
    assert 1000.0 < r2 < 9000.0, r2          # TFLOP/s


def test_probe_rejects_bad_arguments():
    import ctypes

    import routed_expert_ffn_histogram_gb300 as M

    L = M.lib()
    n = ctypes.c_int(0)
    assert L.moe_probe_mxf8f6f4(0, None, ctypes.byref(n), None) == M.MOE_ERR_INVALID
    assert L.moe_probe_mxf8f6f4(1 << 17, ctypes.c_void_p(16), ctypes.byref(n), None) == M.MOE_ERR_INVALID
