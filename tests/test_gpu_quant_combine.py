"""GPU parity of the MXFP8 activation quantisation (codes and scales
bit-exact against the oracle, gathered in grouped order) and of the
weighted combine."""
import numpy as np
import pytest

import moe_synth as S
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wid", [0, 3, 4])
def test_quant_mxfp8_gathered(wid):
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    wl = S.WORKLOADS[wid]
    xb = S.activations_bf16_bits(wl, 0)
    ids, _ = oracle.route(S.logits(wl, 0), wl.top_k)
    _, _, perm, _ = oracle.hist_perm(ids, wl.experts)
    T, H = xb.shape
    A = T * wl.top_k
    x = torch.from_numpy(xb.view(np.int16)).cuda()
    q = torch.empty((A, H), dtype=torch.uint8, device="cuda")
    stride = ((H // 32 + 15) // 16) * 16
    s = torch.zeros((A, stride), dtype=torch.uint8, device="cuda")
    M.moe_quant_mxfp8(x, q, s, perm=torch.from_numpy(perm).cuda(), k=wl.top_k)
    torch.cuda.synchronize()
    qr, sr = oracle.mxfp8_quant(xb)
    src = perm // wl.top_k
    assert np.array_equal(q.cpu().numpy(), qr[src])
    assert np.array_equal(s.cpu().numpy()[:, : H // 32], sr[src])


def test_quant_mxfp8_special_values():
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    rng = np.random.default_rng(4)
    x = torch.from_numpy(rng.standard_normal((16, 256)).astype(np.float32) * 10).to(torch.bfloat16)
    x[0, :32] = 0
    x[1, :32] = -0.0
    x[2, 32:64] = torch.tensor(1e-38)
    x[3, :] = torch.tensor(3e38)
    x[4, 64:96] = torch.tensor(1.75)
    x[4, 65] = 1.8984375
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q = torch.empty((16, 256), dtype=torch.uint8, device="cuda")
    s = torch.empty((16, 8), dtype=torch.uint8, device="cuda")
    M.moe_quant_mxfp8(x.view(torch.int16).cuda(), q, s)
    torch.cuda.synchronize()
    qr, sr = oracle.mxfp8_quant(bits)
    assert np.array_equal(q.cpu().numpy(), qr)
    assert np.array_equal(s.cpu().numpy(), sr)


@pytest.mark.parametrize("T,k,H", [(16, 2, 256), (300, 8, 2048), (5, 1, 12), (3, 4, 2880)])
def test_combine(T, k, H):
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    rng = np.random.default_rng(T + k + H)
    y = rng.standard_normal((T * k, H)).astype(np.float32)
    w = rng.random((T, k)).astype(np.float32)
    perm = rng.permutation(T * k).astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(T * k, dtype=np.int32)
    y_perm = y[perm]
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    M.moe_combine(torch.from_numpy(y_perm).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(inv).cuda(), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.combine(y, w))


def test_quant_mxfp4_bit_exact():
    """MXFP4 activation quantisation (moe_quant_mxfp4, hardware E2M1
    conversion) against the oracle: packed codes and E8M0 scales bit-exact
    on rows spanning 2^-30..2^30 in magnitude, exact ties between E2M1 grid
    points, all-zero blocks, bf16 subnormals and saturating values."""
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    rng = np.random.default_rng(12)
    rows, K = 64, 512
    x = (rng.standard_normal((rows, K)) * np.exp2(rng.integers(-30, 30, (rows, 1)))).astype(np.float32)
    # exact ties: block max 4 (scale 1), the rest on quarter steps of the grid
    x[1, :32] = 4.0
    x[1, 1:32] = np.array([m / 4 for m in range(1, 32)], np.float32) % 6.0
    x[2, 32:64] = 0.0                                  # all-zero block
    x[3, 64:96] = np.float32(1e-40)                    # bf16 subnormals
    x[4, 96:128] = np.linspace(-7.9, 7.9, 32, dtype=np.float32)   # saturates at +-6 after scaling by 1
    x[4, 96] = 7.9
    xt = torch.from_numpy(x).to(torch.bfloat16)
    xb = xt.view(torch.int16).numpy().view(np.uint16)
    q = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    s = torch.zeros((rows, K // 32), dtype=torch.uint8, device="cuda")
    M.moe_quant_mxfp4(xt.cuda(), q, s)
    torch.cuda.synchronize()
    qr, sr = oracle.mxfp4_quant(xb)
    assert np.array_equal(s.cpu().numpy(), sr)
    assert np.array_equal(q.cpu().numpy(), qr)
