"""Pins of the float64 backward oracle (oracle/moe_oracle_grad.py).

The gradients are tied to things other than the backward code itself:
  * central finite differences of the forward oracle's objective on small
    layers, for every element of every input and weight (the routing is
    held at the unperturbed choice, which is what "the top-K choice passes no
    gradient" means, and no token of these layers has a near-tied logit);
  * torch.autograd of a plain expert written out in the test (N = K = 1);
  * invariants of the objective: shifting one token's logits by a constant
    changes only the z-loss; balanced counts make the load-balance gradient
    vanish; with every assignment dropped the layer is the residual;
  * planted mistakes (on the CPU), each of which a pin must catch.
"""
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import moe_oracle_grad as G

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def make_layer(seed, *, T, d, F, N, K, activation="swiglu", has_bias=False,
               router_bias=False, n_shared=0, select_bias=False):
    rng = np.random.default_rng(seed)
    E = N + n_shared
    lay = {
        "x": rng.normal(0, 1.0, (T, d)),
        "w_r": rng.normal(0, 1.0 / math.sqrt(d), (N, d)),
        "b_r": rng.normal(0, 0.3, N) if router_bias else None,
        "dy": rng.normal(0, 1.0, (T, d)),
        "sel": rng.normal(0, 0.5, N) if select_bias else None,
    }
    if activation == "swiglu":
        lay["W"] = {"w_gate": rng.normal(0, 0.4, (E, F, d)),
                    "w_up": rng.normal(0, 0.4, (E, F, d)),
                    "w_down": rng.normal(0, 0.4, (E, d, F))}
    else:
        lay["W"] = {"w1": rng.normal(0, 0.4, (E, F, d)),
                    "b1": rng.normal(0, 0.2, (E, F)) if has_bias else None,
                    "w2": rng.normal(0, 0.4, (E, d, F)),
                    "b2": rng.normal(0, 0.2, (E, d)) if has_bias else None}
    return lay


def expert_of(W):
    return lambda e: {k: v[e] for k, v in W.items() if v is not None}


def common(opts):
    return {k: opts[k] for k in ("K", "activation", "capacity_factor", "alpha", "z_coef",
                                 "add_residual", "gate_mode", "n_shared")}


def objective(lay, opts, idx):
    return G.objective(lay["x"], lay["w_r"], lay["b_r"], expert_of(lay["W"]), lay["dy"],
                       select_bias=lay["sel"], idx_override=idx, **common(opts))


def analytic(lay, opts, **kw):
    return G.moe_backward(lay["x"], lay["w_r"], lay["b_r"], expert_of(lay["W"]), lay["dy"],
                          select_bias=lay["sel"], **common(opts), **kw)


def fd_max_error(lay, opts, h=1e-5):
    """Max over every parameter element of |analytic - central difference|,
    relative to the largest gradient magnitude."""
    g = analytic(lay, opts)
    idx = g["fwd"]["idx"]
    # the routing must not sit near a tie (else the derivative is not defined)
    l = g["fwd"]["logits"] + (0.0 if lay["sel"] is None else lay["sel"][None, :])
    assert not O.near_tie_tokens(l, opts["K"], 1e-3).any()
    pairs = [(lay["x"], g["dx"]), (lay["w_r"], g["dw_r"])]
    if lay["b_r"] is not None:
        pairs.append((lay["b_r"], g["db_r"]))
    for name, arr in lay["W"].items():
        if arr is None:
            continue
        grad = np.stack([g["dw"][e]["d" + name] for e in range(arr.shape[0])])
        pairs.append((arr, grad))
    worst, scale = 0.0, 0.0
    for arr, grad in pairs:
        assert grad.shape == arr.shape
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + h
            lp = objective(lay, opts, idx)
            flat[i] = keep - h
            lm = objective(lay, opts, idx)
            flat[i] = keep
            worst = max(worst, abs((lp - lm) / (2 * h) - gflat[i]))
        scale = max(scale, float(np.max(np.abs(grad), initial=0.0)))
    return worst / max(scale, 1e-30)


BASE = dict(K=2, activation="swiglu", capacity_factor=math.inf, alpha=0.01, z_coef=0.0,
            add_residual=False, gate_mode="renorm", n_shared=0)

FD_CASES = {
    "renorm_uncapped": (dict(T=7, d=6, F=5, N=4), {}),
    "capacity_residual_z_bias": (dict(T=9, d=5, F=4, N=3, router_bias=True),
                                 dict(capacity_factor=0.5, add_residual=True, z_coef=0.3,
                                      alpha=0.2)),
    "switch_gate_top1_selbias_shared": (dict(T=8, d=5, F=3, N=4, n_shared=1, select_bias=True),
                                        dict(K=1, gate_mode="softmax", alpha=0.1,
                                             capacity_factor=1.0, n_shared=1)),
    "gelu_bias_two_shared": (dict(T=6, d=4, F=5, N=3, activation="gelu", has_bias=True,
                                  n_shared=2, router_bias=True),
                             dict(activation="gelu", n_shared=2, capacity_factor=1.0,
                                  z_coef=0.05, alpha=0.3)),
    "dense_k_eq_n": (dict(T=5, d=4, F=3, N=3), dict(K=3, alpha=0.5)),
    "top3_capacity_softmax_gate": (dict(T=10, d=4, F=3, N=5, router_bias=True),
                                   dict(K=3, capacity_factor=0.7, gate_mode="softmax",
                                        alpha=0.1, z_coef=0.2, add_residual=True)),
}


@pytest.mark.parametrize("name", sorted(FD_CASES))
def test_gradients_match_finite_differences(name):
    shape, extra = FD_CASES[name]
    opts = {**BASE, **extra}
    for seed in range(40):  # first seed whose routing has no near-tie
        lay = make_layer(seed, K=opts["K"], **shape)
        l = O.router_logits(lay["x"], lay["w_r"], lay["b_r"])
        if lay["sel"] is not None:
            l = l + lay["sel"][None, :]
        if not O.near_tie_tokens(l, opts["K"], 1e-3).any():
            break
    assert fd_max_error(lay, opts) < 1e-7


def test_capacity_case_drops_assignments():
    """The capacity cases above do exercise drops."""
    shape, extra = FD_CASES["capacity_residual_z_bias"]
    lay = make_layer(0, K=2, **shape)
    g = analytic(lay, {**BASE, **extra})
    assert g["fwd"]["n_dropped"] > 0
    dropped = g["fwd"]["slot_of"] < 0
    assert np.all(g["dg"][dropped] == 0.0)


def test_subsets_equal_full():
    """Returning dx for some tokens / dW for some experts changes nothing."""
    lay = make_layer(3, T=12, d=5, F=4, N=4, K=2, n_shared=1)
    opts = {**BASE, "n_shared": 1, "capacity_factor": 0.8, "add_residual": True}
    full = analytic(lay, opts)
    part = analytic(lay, opts, tokens=[2, 7, 11], experts=[1, 4], router_grads=False)
    assert np.allclose(part["dx"], full["dx"][[2, 7, 11]], rtol=0, atol=1e-13)
    for e in (1, 4):
        for k, v in part["dw"][e].items():
            assert np.allclose(v, full["dw"][e][k], rtol=0, atol=1e-13)


# ------------------------------------------------ autograd of one expert ----
def test_single_expert_swiglu_matches_autograd():
    """N = K = 1: y = E(x) ([替代FFN] §1, the plain FFN); the gradients of
    <dy, E(x)> by torch.autograd on an expert written here."""
    lay = make_layer(5, T=9, d=6, F=7, N=1, K=1)
    opts = {**BASE, "K": 1, "alpha": 0.0}
    g = analytic(lay, opts)
    x = torch.tensor(lay["x"], requires_grad=True)
    wg, wu, wd = (torch.tensor(lay["W"][k][0], requires_grad=True)
                  for k in ("w_gate", "w_up", "w_down"))
    a, b = x @ wg.T, x @ wu.T
    y = (a * torch.sigmoid(a) * b) @ wd.T
    (y * torch.tensor(lay["dy"])).sum().backward()
    assert np.allclose(g["dx"], x.grad.numpy(), rtol=0, atol=1e-12)
    for name, t in (("dw_gate", wg), ("dw_up", wu), ("dw_down", wd)):
        assert np.allclose(g["dw"][0][name], t.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(g["dw_r"], 0.0, atol=1e-15)  # one expert: gate 1, softmax 1


def test_single_expert_gelu_matches_autograd():
    lay = make_layer(6, T=8, d=5, F=6, N=1, K=1, activation="gelu", has_bias=True)
    opts = {**BASE, "K": 1, "alpha": 0.0, "activation": "gelu"}
    g = analytic(lay, opts)
    x = torch.tensor(lay["x"], requires_grad=True)
    w1, b1, w2, b2 = (torch.tensor(lay["W"][k][0], requires_grad=True)
                      for k in ("w1", "b1", "w2", "b2"))
    y = torch.nn.functional.gelu(x @ w1.T + b1) @ w2.T + b2
    (y * torch.tensor(lay["dy"])).sum().backward()
    assert np.allclose(g["dx"], x.grad.numpy(), rtol=0, atol=1e-12)
    for name, t in (("dw1", w1), ("db1", b1), ("dw2", w2), ("db2", b2)):
        assert np.allclose(g["dw"][0][name], t.grad.numpy(), rtol=0, atol=1e-12)


# ------------------------------------------------------------ invariants ----
def test_logit_shift_only_moves_z_loss():
    """Adding c to all of a token's logits leaves the gates, p and the
    selection unchanged and adds 2 c lse_t / T-terms only through the z-loss:
    sum_e dL/dl[t, e] = z_coef * 2 * lse_t / T."""
    lay = make_layer(7, T=20, d=6, F=4, N=6, K=2, router_bias=True)
    for gm in ("renorm", "softmax"):
        opts = {**BASE, "gate_mode": gm, "alpha": 0.3, "z_coef": 0.7, "capacity_factor": 1.0}
        g = analytic(lay, opts)
        l = g["fwd"]["logits"]
        m = l.max(axis=1)
        lse = m + np.log(np.exp(l - m[:, None]).sum(axis=1))
        T = l.shape[0]
        assert np.allclose(g["dl"].sum(axis=1), 0.7 * 2 * lse / T, rtol=0, atol=1e-13)
        assert abs(g["db_r"].sum() - 0.7 * 2 * lse.sum() / T) < 1e-12


def test_balanced_counts_zero_aux_gradient():
    """With f_e = 1/N for every expert, sum_e f_e P_e = 1/N whatever p is, so
    L_aux has zero gradient: cyclically rotated logits, dy = 0, no z-loss."""
    N, K, m = 4, 2, 3
    T, d = m * N, N
    base = np.array([3.0, 1.0, 0.0, -2.0])
    x = np.stack([np.roll(base, t % N) for t in range(T)])
    w_r = np.eye(N)
    W = make_layer(0, T=T, d=d, F=3, N=N, K=K)["W"]
    g = G.moe_backward(x, w_r, None, expert_of(W), np.zeros((T, d)), K=K,
                       activation="swiglu", alpha=0.5)
    assert np.allclose(g["fwd"]["f"], 1.0 / N)
    assert np.max(np.abs(g["dl"])) < 1e-15 and np.max(np.abs(g["dw_r"])) < 1e-15


def test_everything_dropped_is_residual():
    """C = 0 (CF tiny): no expert output reaches y, so with alpha = z = 0
    the gradient is dx = dy and every weight gradient is zero."""
    lay = make_layer(8, T=6, d=4, F=3, N=4, K=2)
    opts = {**BASE, "capacity_factor": 0.01, "alpha": 0.0, "add_residual": True}
    g = analytic(lay, opts)
    assert g["fwd"]["C"] == 0
    assert np.array_equal(g["dx"], lay["dy"])
    assert all(np.all(v == 0) for e in g["dw"] for v in g["dw"][e].values())
    assert np.all(g["dw_r"] == 0)


# ------------------------------------------------------- planted mistakes ----
MUTANT_CASE = ("capacity_residual_z_bias", 0)


def mutant_error(monkeypatch, target, replacement, case=None):
    name, seed = case or MUTANT_CASE
    shape, extra = FD_CASES[name]
    opts = {**BASE, **extra}
    lay = make_layer(seed, K=opts["K"], **shape)
    monkeypatch.setattr(target[0], target[1], replacement)
    return fd_max_error(lay, opts)


def test_mutant_silu_grad_missing_term(monkeypatch):
    def wrong(a):
        return 1.0 / (1.0 + np.exp(-a))  # drops the a * (1 - sigmoid) term
    assert mutant_error(monkeypatch, (G, "silu_grad"), wrong) > 1e-3


def test_mutant_gelu_grad_cdf_only(monkeypatch):
    def wrong(z):
        return 0.5 * (1.0 + G._erf(z / math.sqrt(2.0)))
    assert mutant_error(monkeypatch, (G, "gelu_erf_grad"), wrong,
                        ("gelu_bias_two_shared", 0)) > 1e-3


def test_mutant_aux_term_dropped(monkeypatch):
    real = G.logit_grad

    def wrong(l, idx, gate, dg, f, *, alpha, z_coef, gate_mode):
        return real(l, idx, gate, dg, f, alpha=0.0, z_coef=z_coef, gate_mode=gate_mode)
    assert mutant_error(monkeypatch, (G, "logit_grad"), wrong) > 1e-3


def test_mutant_z_term_dropped(monkeypatch):
    real = G.logit_grad

    def wrong(l, idx, gate, dg, f, *, alpha, z_coef, gate_mode):
        return real(l, idx, gate, dg, f, alpha=alpha, z_coef=0.0, gate_mode=gate_mode)
    assert mutant_error(monkeypatch, (G, "logit_grad"), wrong) > 1e-3


def test_mutant_renorm_gate_treated_as_softmax(monkeypatch):
    real = G.logit_grad

    def wrong(l, idx, gate, dg, f, *, alpha, z_coef, gate_mode):
        return real(l, idx, gate, dg, f, alpha=alpha, z_coef=z_coef, gate_mode="softmax")
    assert mutant_error(monkeypatch, (G, "logit_grad"), wrong) > 1e-3


def test_mutant_up_gradient_uses_gate_branch(monkeypatch):
    real = G.expert_backward_swiglu

    def wrong(xe, w_gate, w_up, w_down, do):
        out = real(xe, w_gate, w_up, w_down, do)
        out["dw_up"] = out["dw_gate"]
        return out
    assert mutant_error(monkeypatch, (G, "expert_backward_swiglu"), wrong) > 1e-3


def test_mutant_gate_applied_twice(monkeypatch):
    """The expert output gradient scaled once more by a gate-sized factor."""
    real = G.expert_backward

    def wrong(activation, xe, ew, do):
        return real(activation, xe, ew, 0.5 * do)
    assert mutant_error(monkeypatch, (G, "expert_backward"), wrong) > 1e-3
