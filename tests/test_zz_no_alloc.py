"""moe_route_no_workspace: the router for callers that cannot allocate device
memory (a serving process whose device memory is all owned by its own pool, a
plug-in interface with no workspace argument). Its results are checked
against the float64 oracle (routing, gates, counts, f, P, L_aux) and against
moe_route, which takes a caller workspace, on consecutive calls that share
its fixed scratch array; requests at and just past the array's limit are
checked too.

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


def route(w, inp, use_ws):
    cfg = moe.LayerConfig.from_workload(w)
    T, K, N = w.T, w.K, w.N
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    gate = torch.zeros((T, K), dtype=torch.float32, device="cuda")
    st = moe.Stats(N)
    if use_ws:
        moe.moe_route(cfg, inp["x"], inp["w_r"], inp["b_r"], idx, gate, st,
                      moe.alloc_workspace(cfg))
    else:
        moe.moe_route_no_workspace(cfg, inp["x"], inp["w_r"], inp["b_r"], idx, gate, st)
    torch.cuda.synchronize()
    return idx.cpu().numpy().astype(np.int64), gate.cpu().numpy(), st.to_host()


def logits64(inp):
    return O.router_logits(inp["x"].cpu(), inp["w_r"].cpu(),
                           None if inp["b_r"] is None else inp["b_r"].cpu())


def assert_matches_oracle(w, l64, out):
    """Routing bit-exact except near-tie tokens; gates, counts, f, P and L_aux
    of the oracle on the GPU's routing, within the parity tests' bars."""
    idx, gate, st = out
    L.check_routing(l64, idx, w.K)
    assert np.max(np.abs(gate - O.renormalised_gates(l64, idx)), initial=0) <= L.GATE_TOL
    count, f, P, l_aux = O.load_balance(idx, O.softmax(l64), w.N, w.alpha)
    assert np.array_equal(st["count"], count)
    assert np.allclose(st["f"], f, rtol=1e-6, atol=0)
    assert np.allclose(st["P"], P, rtol=L.STAT_RTOL, atol=1e-7)
    assert abs(st["l_aux"] - l_aux) <= L.STAT_RTOL * abs(l_aux) + 1e-9
    assert st["status"] == 0


def assert_matches_moe_route(w, l64, a, b):
    """The bar between the two entry points: indices agree except on near-tie
    tokens (each differing choice within 1e-5 in float64 logit); gates on the
    agreeing tokens, P and L_aux within their tolerances; counts and f equal
    when the routing agrees everywhere, else each call's f is its own count
    over T*K."""
    (ia, ga, sa), (ib, gb, sb) = a, b
    diff = np.any(ia != ib, axis=1)
    assert not np.any(diff & ~O.near_tie_tokens(l64, w.K, L.NEAR_TIE_EPS))
    for t in np.nonzero(diff)[0]:
        assert np.all(np.abs(l64[t, ia[t]] - l64[t, ib[t]]) < L.NEAR_TIE_EPS)
    same = ~diff
    assert np.max(np.abs(ga[same] - gb[same]), initial=0) <= L.GATE_TOL
    if not diff.any():
        assert np.array_equal(sa["count"], sb["count"])
        assert np.array_equal(sa["f"], sb["f"])
    for s in (sa, sb):
        assert np.allclose(s["f"], s["count"] / float(w.T * w.K), rtol=1e-6, atol=0)
    assert np.allclose(sa["P"], sb["P"], rtol=L.STAT_RTOL, atol=1e-7)
    assert abs(sa["l_aux"] - sb["l_aux"]) <= L.STAT_RTOL * abs(sa["l_aux"]) + 1e-9
    assert sa["status"] == sb["status"] == 0


LAYERS = [
    # bf16 with d % 64 == 0: moe_route takes the tensor-core router here
    MoEWorkload("no_alloc_bf16", T=4096, d=1024, F=128, N=64, K=2, router_bias="skew"),
    # fp32 (both entry points on the CUDA-core router)
    MoEWorkload("no_alloc_fp32", T=1000, d=100, F=4, N=8, K=1, dtype="f32", init="uniform",
                router_bias="uniform"),
    MoEWorkload("no_alloc_bf16_small", T=777, d=512, F=128, N=8, K=2),
]


def test_matches_oracle_and_moe_route_on_calls_in_a_row():
    # different layers back to back: no call may see the previous call's
    # leftovers in the shared scratch array
    for w in LAYERS:
        inp = L.device_inputs(w)
        l64 = logits64(inp)
        with_ws = route(w, inp, True)
        without_ws = route(w, inp, False)
        assert_matches_oracle(w, l64, without_ws)
        assert_matches_moe_route(w, l64, with_ws, without_ws)


def test_largest_request_at_the_limit_and_one_token_past_it():
    # ceil(T / 32) * (N + 2) <= 131072 at N = 256: T = 16256 is the largest
    # accepted batch (508 blocks * 258 = 131064); T = 16257 needs 509 blocks
    w = MoEWorkload("no_alloc_limit", T=16256, d=256, F=128, N=256, K=8)
    inp = L.device_inputs(w)
    l64 = logits64(inp)
    out = route(w, inp, False)
    assert_matches_oracle(w, l64, out)
    again = route(w, inp, False)  # a second call on the same scratch: same bits
    for a, b in zip(out[:2], again[:2]):
        assert np.array_equal(a, b)
    assert np.array_equal(out[2]["P"], again[2]["P"])

    past = MoEWorkload("no_alloc_past", T=16257, d=256, F=128, N=256, K=8)
    cfg = moe.LayerConfig.from_workload(past)
    x = torch.zeros((past.T, 256), dtype=torch.bfloat16, device="cuda")
    w_r = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    idx = torch.full((past.T, 8), -3, dtype=torch.int32, device="cuda")
    gate = torch.zeros((past.T, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_route_no_workspace(cfg, x, w_r, None, idx, gate, None)
    assert e.value.code == moe.moe.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (idx == -3).all()  # rejected before anything was launched
