"""GPU parity of moe_route_plan against the oracle: ids, counts, offsets,
perm and inv bit-exact; routing weights within 2 ulp."""
import numpy as np
import pytest

import moe_synth as S
import oracle
from helpers import ULP_TOL_W, f32_ulp_diff

pytestmark = pytest.mark.gpu


def _run(logits, k, counts_host=True):
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    T, E = logits.shape
    lg = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    plan = M.RoutePlan.allocate(T, E, k, counts_host=counts_host)
    M.moe_route_plan(lg, k, plan, with_counts_host=counts_host)
    torch.cuda.synchronize()
    n = T * k
    res = dict(ids=plan.ids.cpu().numpy(), w=plan.w.cpu().numpy(), counts=plan.counts.cpu().numpy(),
               offsets=plan.offsets.cpu().numpy(), perm=plan.perm.cpu().numpy()[:n],
               inv=plan.inv.cpu().numpy()[:n])
    if counts_host:
        res["counts_host"] = plan.counts_host.numpy().copy()
    return res


def _check(logits, k):
    E = logits.shape[1]
    got = _run(logits, k)
    ids, w = oracle.route(logits, k)
    counts, offsets, perm, inv = oracle.hist_perm(ids, E)
    assert np.array_equal(got["ids"], ids)
    assert np.all(f32_ulp_diff(got["w"], w) <= ULP_TOL_W)
    assert np.array_equal(got["counts"], counts)
    assert np.array_equal(got["counts_host"], counts)
    assert np.array_equal(got["offsets"], offsets)
    assert np.array_equal(got["perm"], perm)
    assert np.array_equal(got["inv"], inv)
    return got


@pytest.mark.parametrize("wid", [0, 1, 2, 3, 4])
def test_route_workloads(wid):
    wl = S.WORKLOADS[wid]
    for layer, step in [(0, 0), (wl.layers - 1, wl.steps - 1)]:
        got = _check(S.logits(wl, layer, step), wl.top_k)
    if wid == 3:
        assert int((got["counts"] > 0).sum()) == 32  # each unique expert once, 32 per layer


@pytest.mark.parametrize("T,E,k", [(1, 8, 1), (1, 8, 8), (5, 32, 32), (37, 8, 3), (257, 16, 2), (300, 256, 8),
                                   (1000, 7, 7), (513, 130, 5)])
def test_route_shapes(T, E, k):
    rng = np.random.default_rng(T * 31 + E * 7 + k)
    _check(rng.standard_normal((T, E)).astype(np.float32), k)


def test_route_ties_and_empty_groups():
    rng = np.random.default_rng(9)
    lg = np.round(rng.standard_normal((600, 32)) * 1.5).astype(np.float32)
    lg[:, 5] = -50.0  # expert 5 never chosen: an empty group
    lg[0, :] = 0.0
    lg[1, :] = -0.0
    got = _check(lg, 4)
    assert got["counts"][5] == 0
    assert got["ids"][0].tolist() == [0, 1, 2, 3]


def test_route_zero_tokens():
    import torch

    import routed_expert_ffn_histogram_gb300 as M

    plan = M.RoutePlan.allocate(0, 8, 2)
    plan.counts.fill_(7)
    M.moe_route_plan(torch.empty((0, 8), device="cuda"), 2, plan, with_counts_host=False)
    torch.cuda.synchronize()
    assert plan.counts.cpu().tolist() == [0] * 8 and plan.offsets.cpu().tolist() == [0] * 9


def test_route_repeatable():
    wl = S.WORKLOADS[4]
    lg = S.logits(wl, 0)
    a, b = _run(lg, wl.top_k), _run(lg, wl.top_k)
    for key in a:
        assert np.array_equal(a[key], b[key])
