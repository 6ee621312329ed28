"""GPU parity of the backward pass (moe_backward through the C ABI) against
the float64 backward oracle (oracle/moe_oracle_grad.py).

Each case runs moe_forward with save_for_backward, then moe_backward with a
seeded output gradient dy, and compares every gradient element by element
with the oracle evaluated on the GPU's routing (the routing itself is checked
against the oracle first). Bars: max |err| <= 1e-4 * rms for fp32 layers;
for bf16 layers every element within the first-order bound of the bf16
roundings the backward performs (moe_testlib.grad_rounding_bounds), per
gradient tensor and per expert.
"""
import numpy as np
import pytest
import torch

import moe_inputs
from moe_inputs import MoEWorkload

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mixture_experts_layer_101_b300 as moe
    import moe_testlib as L


def wl(name="case", **kw):
    base = dict(T=100, d=256, F=128, N=4, K=2)
    base.update(kw)
    return MoEWorkload(name, **base)


CASES = {
    # bf16 SwiGLU on the tensor-core forward; several row tiles per expert
    "bf16_top2": (wl(T=300, d=256, F=256, N=3, K=2), 0.0),
    "bf16_top8_of_64": (wl(T=257, d=512, F=256, N=64, K=8), 0.0),
    "bf16_capacity_residual_z": (wl(T=1000, d=256, F=128, N=8, K=1, capacity_factor=1.25,
                                    add_residual=True, router_bias="skew"), 0.1),
    "bf16_softmax_gate_selbias_shared": (wl(T=400, d=256, F=128, N=16, K=2, gate_mode="softmax",
                                            select_bias="uniform", n_shared=1,
                                            router_bias="uniform"), 0.05),
    "bf16_one_token": (wl(T=1, d=256, F=128, N=8, K=2), 0.0),
    "bf16_odd_shapes": (wl(T=150, d=72, F=100, N=6, K=2), 0.2),  # CUDA-core forward
    "bf16_two_shared_capacity": (wl(T=600, d=512, F=128, N=16, K=2, n_shared=2,
                                    capacity_factor=0.5, add_residual=True), 0.0),
    # long per-expert reductions with ragged tails; 128-column tiles along F
    "bf16_many_rows_f384": (wl(T=3000, d=256, F=384, N=2, K=1, router_bias="uniform"), 0.0),
    # backward products on CTA pairs (>= 512 rows per expert): skewed counts,
    # drops, ragged padded tails
    "bf16_pairs_capacity_skew": (wl(T=3000, d=512, F=512, N=4, K=2, capacity_factor=0.9,
                                    router_bias="skew"), 0.0),
    # forward GEMMs as CTA pairs, expert tails of 244 241 3 24 rows past whole
    # 256-row pair tiles
    "bf16_pair_tails_mixed": (wl(T=2048, d=1024, F=1024, N=4, K=2, router_bias="uniform"), 0.0),
    # decode-sized batch: the forward's split gate/up reduction keeps the
    # pre-activations through its combining kernel
    "bf16_decode_split_k": (wl(T=24, d=1024, F=256, N=8, K=2), 0.0),
    # forward on CTA pairs (pre-activations kept by the pair kernel)
    "bf16_pair_forward_shared": (wl(T=2048, d=1024, F=2048, N=2, K=1, n_shared=1,
                                    capacity_factor=1.5, add_residual=True), 0.0),
    # fp32 layers (CUDA-core forward), GELU with bias
    "f32_gelu_bias": (wl(T=64, d=64, F=128, N=4, K=2, dtype="f32", activation="gelu",
                         has_bias=True, init="uniform", router_bias="uniform"), 0.0),
    "f32_gelu_capacity_residual_z": (wl(T=128, d=64, F=128, N=4, K=2, dtype="f32",
                                        activation="gelu", has_bias=True, init="uniform",
                                        router_bias="uniform", capacity_factor=0.5,
                                        add_residual=True), 0.3),
    "f32_swiglu_k3": (wl(T=77, d=36, F=52, N=5, K=3, dtype="f32", init="uniform"), 0.0),
    "f32_gelu_nobias_shared_softmax": (wl(T=90, d=64, F=96, N=4, K=2, dtype="f32",
                                          activation="gelu", init="uniform", n_shared=2,
                                          gate_mode="softmax"), 0.02),
    "f32_dense_k_eq_n": (wl(T=50, d=32, F=40, N=4, K=4, dtype="f32", init="uniform",
                            alpha=0.5), 0.0),
}


def inputs(w):
    inp = L.device_inputs(w)
    cfg = L.layer_config(w, inp)
    dy = moe_inputs.make_dy(w).cuda()
    return cfg, inp, dy


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_small(name):
    w, z = CASES[name]
    cfg, inp, dy = inputs(w)
    ratios = L.check_backward(cfg, inp, dy, z)
    print(name, {k: f"{v:.2e}" for k, v in ratios.items()})


# Full-size layers in the configuration the training bench times: dx on
# sampled tokens (every assignment of each, including dropped ones), the
# weight gradients of sampled experts (hot and cold), and the router
# gradients where the oracle can afford every expert row (Switch, decode).
FULL = {
    "switch_skewed": dict(experts=[0, 37], router_grads=True),
    "mixtral_decode": dict(experts=None, router_grads=True),
    "mixtral_prefill": dict(experts=[], router_grads=False),
    "deepseek_fine": dict(experts=[5, 200], router_grads=False),
    "deepseek_shared": dict(experts=[17, 256], router_grads=False),
}


@pytest.mark.parametrize("name", sorted(FULL))
def test_backward_full_size(name):
    w = moe_inputs.WORKLOADS[name]
    cfg, inp, dy = inputs(w)
    rng = np.random.default_rng(11)
    tokens = sorted(rng.choice(w.T, size=min(w.T, 40), replace=False).tolist())
    ratios = L.check_backward(cfg, inp, dy, 1e-3, tokens=tokens, **FULL[name])
    print(name, {k: f"{v:.2e}" for k, v in ratios.items()})


def test_backward_deterministic():
    w, z = CASES["bf16_capacity_residual_z"]
    cfg, inp, dy = inputs(w)
    g1, _, _, _ = L.run_backward(cfg, inp, dy, z)
    g2, _, _, _ = L.run_backward(cfg, inp, dy, z)
    for k, v in g1.items():
        if v is not None:
            assert torch.equal(v, g2[k]), k


@pytest.mark.parametrize("name", ["bf16_capacity_residual_z", "bf16_pair_tails_mixed"])
def test_training_step_graph_replay(name):
    """forward + backward captured as one CUDA graph and replayed after new x
    and dy are copied into their buffers gives the same bits as the eager
    calls on the new data."""
    w, z = CASES[name]
    cfg, inp, dy = inputs(w)
    cfg.save_for_backward = True
    layer = moe.MoELayer(cfg, inp["w_r"], inp["b_r"], inp["experts"])
    xbuf, dybuf = inp["x"].clone(), dy.clone()
    grads = moe.alloc_grads(cfg, inp["b_r"] is not None)

    def step():
        layer.forward(xbuf)
        layer.backward(dybuf, z, grads)

    graph = moe.capture_graph(step)
    x2 = (inp["x"].float() * -0.75).to(inp["x"].dtype)
    dy2 = (dy.float() * 1.5).to(dy.dtype)
    xbuf.copy_(x2)
    dybuf.copy_(dy2)
    graph.replay()
    torch.cuda.synchronize()
    g_graph = {k: v.clone() for k, v in grads.items() if v is not None}
    y_graph = layer.y.clone()
    layer.forward(x2)
    layer.backward(dy2, z, grads)
    torch.cuda.synchronize()
    assert torch.equal(y_graph, layer.y)
    for k, v in g_graph.items():
        assert torch.equal(v, grads[k]), k
    assert layer.stats.to_host()["status"] == 0


def test_backward_needs_saved_state():
    w, _ = CASES["bf16_top2"]
    cfg, inp, dy = inputs(w)
    layer = moe.MoELayer(cfg, inp["w_r"], inp["b_r"], inp["experts"])  # no save_for_backward
    layer.forward(inp["x"])
    with pytest.raises(moe.MoEError) as ei:
        layer.backward(dy)
    assert ei.value.code == moe.moe.MOE_ERR_INVALID


def test_backward_rejects_bad_z_coef():
    w, _ = CASES["bf16_top2"]
    cfg, inp, dy = inputs(w)
    cfg.save_for_backward = True
    layer = moe.MoELayer(cfg, inp["w_r"], inp["b_r"], inp["experts"])
    layer.forward(inp["x"])
    for z in (-1.0, float("nan"), float("inf")):
        with pytest.raises(moe.MoEError) as ei:
            layer.backward(dy, z)
        assert ei.value.code == moe.moe.MOE_ERR_INVALID


def test_backward_zero_tokens_gives_zero_gradients():
    """T = 0: every gradient buffer is written with zeros (the buffers start
    filled with NaN)."""
    base = wl(T=1, d=256, F=128, N=4, K=2)
    inp = L.device_inputs(base)
    cfg = moe.LayerConfig.from_workload(base, T=0)
    cfg.save_for_backward = True
    layer = moe.MoELayer(cfg, inp["w_r"], inp["b_r"], inp["experts"])
    layer.forward(inp["x"])  # a valid pointer; no row of it is read
    grads = moe.alloc_grads(cfg, router_bias=True)
    for v in grads.values():
        if v is not None:
            v.fill_(float("nan"))
    g = layer.backward(moe_inputs.make_dy(base).cuda(), grads=grads)
    torch.cuda.synchronize()
    for k, v in g.items():
        if v is not None and v.numel() > 0:
            assert torch.count_nonzero(v) == 0, k
