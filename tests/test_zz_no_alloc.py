"""moe_route_no_workspace: the router for callers that cannot allocate
device memory (a serving process whose device memory is all owned by its own
pool, a plug-in interface with no workspace argument). It must give the
results of moe_route, which takes a caller workspace, and keep giving them
on consecutive calls that share its fixed scratch array.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

from moe_inputs import MoEWorkload
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mixture_experts_layer_101_b300 as moe
    import moe_testlib as L


def route_both_ways(w):
    cfg = moe.LayerConfig.from_workload(w)
    inp = L.device_inputs(w)
    T, K, N = w.T, w.K, w.N
    outs = []
    for use_ws in (True, False):
        idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
        gate = torch.zeros((T, K), dtype=torch.float32, device="cuda")
        st = moe.Stats(N)
        if use_ws:
            moe.moe_route(cfg, inp["x"], inp["w_r"], inp["b_r"], idx, gate, st,
                          moe.alloc_workspace(cfg))
        else:
            moe.moe_route_no_workspace(cfg, inp["x"], inp["w_r"], inp["b_r"], idx, gate, st)
        torch.cuda.synchronize()
        outs.append((idx.cpu().numpy(), gate.cpu().numpy(), st.to_host()))
    l64 = O.router_logits(inp["x"].cpu(), inp["w_r"].cpu(),
                          None if inp["b_r"] is None else inp["b_r"].cpu())
    return outs, l64


def assert_same(a, b, l64, K):
    """The routing bar of the parity tests: indices agree except on near-tie
    tokens (each differing choice within 1e-5 in float64 logit); gates, P and
    L_aux within their tolerances."""
    (ia, ga, sa), (ib, gb, sb) = a, b
    diff = np.any(ia != ib, axis=1)
    assert not np.any(diff & ~O.near_tie_tokens(l64, K, L.NEAR_TIE_EPS))
    for t in np.nonzero(diff)[0]:
        assert np.all(np.abs(l64[t, ia[t]] - l64[t, ib[t]]) < L.NEAR_TIE_EPS)
    same = ~diff
    assert np.max(np.abs(ga[same] - gb[same]), initial=0) <= L.GATE_TOL
    if not diff.any():
        assert np.array_equal(sa["count"], sb["count"])
    assert np.allclose(sa["f"], sb["f"], rtol=1e-6, atol=0)
    assert np.allclose(sa["P"], sb["P"], rtol=L.STAT_RTOL, atol=1e-7)
    assert abs(sa["l_aux"] - sb["l_aux"]) <= L.STAT_RTOL * abs(sa["l_aux"]) + 1e-9
    assert sa["status"] == sb["status"] == 0


def test_matches_moe_route_on_two_calls_in_a_row():
    # two different layers back to back: the second call must not see the
    # first call's leftovers in the shared scratch array
    first = MoEWorkload("no_alloc_a", T=4096, d=1024, F=128, N=64, K=2, router_bias="skew")
    second = MoEWorkload("no_alloc_b", T=1000, d=512, F=128, N=8, K=1)
    for w in (first, second):
        (with_ws, without_ws), l64 = route_both_ways(w)
        assert_same(with_ws, without_ws, l64, w.K)


def test_rejects_requests_beyond_the_scratch_limit():
    w = MoEWorkload("too_big", T=16385, d=256, F=128, N=256, K=8)  # ceil(T/32)*N > 131072
    cfg = moe.LayerConfig.from_workload(w)
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device="cuda")
    w_r = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    idx = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    gate = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_route_no_workspace(cfg, x, w_r, None, idx, gate, None)
    assert e.value.code == moe.moe.MOE_ERR_WORKSPACE
