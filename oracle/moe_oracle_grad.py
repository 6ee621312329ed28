"""Float64 CPU oracle of the backward pass of the sparse Mixture-of-Experts
layer: the gradients of a training objective with respect to the layer's
input, router and expert weights.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
run this module: only the tests, the smoke check of the package entry file
and the CPU-baseline / reference legs of the benchmark script use it. It
shares no code with the CUDA path.

The objective is
    L = sum_{t,j} dy[t,j] * y[t,j] + L_aux + z_coef * z_loss
with dy the gradient of a downstream loss with respect to the layer output
y, L_aux = alpha * N * sum_e f_e * P_e the load-balance loss that training
adds to its objective ([MoE核心思想] 辅助损失公式; [稀疏激活原理] §2.2) and
z_loss the router z-loss ([MoE核心思想] Router Z-Loss; the reading of
moe_oracle.router_z_loss: mean over tokens of the squared log-sum-exp).
Every gradient is the plain derivative of the forward layer of
moe_oracle.moe_forward, written out by the chain rule in float64.

Readings (the pages name the training setting, not its derivatives):
  * the top-K choice, the capacity truncation and the selection bias are
    piecewise constant in the inputs: they pass no gradient. [稀疏激活原理]
    §四 训练不稳定性 states that the expert choice (torch.topk) has zero
    gradient while the gate softmax is differentiable; [概念卡] 结构 4 states
    that the selection bias is adjusted by counting, not by gradients;
  * f_e is a count ("离散统计量", [稀疏激活原理] §2.2) and passes no gradient;
    P_e (continuous) carries the gradient of L_aux into the router;
  * a dropped assignment adds nothing to y, so neither its gate nor its
    expert receives gradient from it;
  * the router receives gradient through the gates, P and the z-loss
    ([概念卡] 结构 2: the router is trained end to end with the model);
  * shared experts have gate 1 and receive dy unchanged.
Pinned by tests/test_oracle_grad_pins.py against central finite differences
of moe_oracle.moe_forward on small layers (every parameter element), against
closed forms and by planted mistakes that the pins must catch.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

from oracle import moe_oracle as O

f64 = O.f64


# --------------------------------------------------------------------------
# experts: derivatives of [稀疏激活原理] §三 class Expert (SwiGLU) and of the
# GELU FFN of [概念卡] 运行示例 / [替代FFN] §1
# --------------------------------------------------------------------------
def silu_grad(a: np.ndarray) -> np.ndarray:
    """d/da [a * sigmoid(a)] = sigmoid(a) * (1 + a * (1 - sigmoid(a)))."""
    s = 1.0 / (1.0 + np.exp(-a))
    return s * (1.0 + a * (1.0 - s))


def gelu_erf_grad(z: np.ndarray) -> np.ndarray:
    """d/dz [z * Phi(z)] = Phi(z) + z * phi(z) (exact-erf GELU)."""
    cdf = 0.5 * (1.0 + _erf(z / math.sqrt(2.0)))
    pdf = np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)
    return cdf + z * pdf


def expert_backward_swiglu(xe, w_gate, w_up, w_down, do) -> dict:
    """Rows xe [R][d], output gradient do [R][d] of o = h W_down^T with
    h = silu(a) * b, a = xe W_gate^T, b = xe W_up^T. Returns dx [R][d] and
    the weight gradients summed over the rows."""
    xe, wg, wu, wd, do = f64(xe), f64(w_gate), f64(w_up), f64(w_down), f64(do)
    a = xe @ wg.T
    b = xe @ wu.T
    h = O.silu(a) * b
    dh = do @ wd                       # [R][F]
    da = dh * b * silu_grad(a)
    db = dh * O.silu(a)
    return {"dx": da @ wg + db @ wu,
            "dw_gate": da.T @ xe, "dw_up": db.T @ xe, "dw_down": do.T @ h}


def expert_backward_gelu(xe, w1, b1, w2, b2, do) -> dict:
    """Rows xe [R][d], output gradient do of o = gelu(z) W2^T (+ b2) with
    z = xe W1^T (+ b1)."""
    xe, w1, w2, do = f64(xe), f64(w1), f64(w2), f64(do)
    z = xe @ w1.T + (f64(b1)[None, :] if b1 is not None else 0.0)
    h = O.gelu_erf(z)
    dh = do @ w2
    dz = dh * gelu_erf_grad(z)
    out = {"dx": dz @ w1, "dw1": dz.T @ xe, "dw2": do.T @ h}
    if b1 is not None:
        out["db1"] = dz.sum(axis=0)
    if b2 is not None:
        out["db2"] = do.sum(axis=0)
    return out


def expert_backward(activation: str, xe, ew: dict, do) -> dict:
    if activation == "swiglu":
        return expert_backward_swiglu(xe, ew["w_gate"], ew["w_up"], ew["w_down"], do)
    return expert_backward_gelu(xe, ew["w1"], ew.get("b1"), ew["w2"], ew.get("b2"), do)


# --------------------------------------------------------------------------
# router: derivatives of the gates ([概念卡] 结构 3; [稀疏激活原理] §三
# MoERouter.forward), of P in L_aux (§2.2) and of the z-loss
# --------------------------------------------------------------------------
def logit_grad(l: np.ndarray, idx: np.ndarray, gate: np.ndarray, dg: np.ndarray,
               f: np.ndarray, *, alpha: float, z_coef: float, gate_mode: str) -> np.ndarray:
    """dL/dl [T][N] for the logits l [T][N], given dL/dgate dg [T][K] (zero
    for dropped assignments) and the assignment fractions f [N].

    renorm gates g_k = exp(l_{i_k}) / sum_k' exp(l_{i_k'}):
        dl_{i_k} += g_k * (dg_k - sum_k' g_k' dg_k');
    softmax gates g_k = p_{i_k}: dp_{i_k} += dg_k;
    L_aux = alpha N sum_e f_e (1/T) sum_t p_te:  dp_te += alpha N f_e / T;
    z_loss = (1/T) sum_t lse_t^2:               dl_t += z_coef (2 lse_t / T) p_t;
    through p = softmax(l):                       dl_t += p_t * (dp_t - <p_t, dp_t>)."""
    T, N = l.shape
    if T == 0:
        return np.zeros((0, N))
    p = O.softmax(l)
    dp = np.zeros((T, N))
    dl = np.zeros((T, N))
    rows = np.arange(T)[:, None]
    if gate_mode == "renorm":
        s = np.sum(gate * dg, axis=1, keepdims=True)
        np.add.at(dl, (np.broadcast_to(rows, idx.shape), idx), gate * (dg - s))
    else:
        np.add.at(dp, (np.broadcast_to(rows, idx.shape), idx), dg)
    dp += alpha * N * f[None, :] / T
    m = l.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(l - m).sum(axis=1))
    dl += z_coef * (2.0 * lse / T)[:, None] * p
    dl += p * (dp - np.sum(p * dp, axis=1, keepdims=True))
    return dl


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------
def moe_backward(x, w_r, b_r, expert_of, dy, *, K: int, activation: str,
                 capacity_factor: float = math.inf, alpha: float = 0.01,
                 z_coef: float = 0.0, add_residual: bool = False,
                 gate_mode: str = "renorm", select_bias=None, n_shared: int = 0,
                 idx_override=None, tokens=None, experts=None,
                 router_grads: bool = True) -> dict:
    """Gradients of L (module docstring) in float64.

    expert_of(e) returns expert e's weights (routed e < N, shared N..N+S-1).
    tokens: the tokens whose dx is returned (None = all); experts: the
    experts (routed or shared indices) whose weight gradients are returned
    (None = all N + n_shared). router_grads: also return dw_r / db_r, which
    need the gate gradient of every token (so every kept expert row).
    idx_override: routing to follow (a GPU choice among near-tied logits).
    Returns dx [len(tokens)][d], dw {e: {name: array}}, dw_r [N][d],
    db_r [N] (if b_r is not None), dl [T][N] and dg [T][K] (when computed for
    all tokens), and the forward dict as "fwd"."""
    xs = f64(x)
    dys = f64(dy)
    T, d = xs.shape
    fwd = O.moe_forward(x, w_r, b_r, expert_of, K=K, activation=activation,
                        capacity_factor=capacity_factor, alpha=alpha,
                        add_residual=add_residual, tokens=[], idx_override=idx_override,
                        gate_mode=gate_mode, select_bias=select_bias, n_shared=n_shared)
    l, idx, gate, f = fwd["logits"], fwd["idx"], fwd["gate"], fwd["f"]
    slot_of = fwd["slot_of"]
    N = l.shape[1]
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    exps = list(range(N + n_shared)) if experts is None else [int(e) for e in experts]
    need_all_dg = router_grads or tokens is None

    # rows each expert must evaluate: all of its kept rows if its weight
    # gradient is wanted or the gate gradient of every token is, else only
    # the requested tokens' rows
    tok_set = set(tok.tolist())
    rows_of = {}
    for t in range(T):
        for k in range(K):
            if slot_of[t, k] < 0:
                continue
            e = int(idx[t, k])
            if need_all_dg or e in exps or t in tok_set:
                rows_of.setdefault(e, []).append((t, k))
    dg = np.zeros((T, K))
    dx_rows = {}  # token -> summed expert input gradient
    dw = {}
    for e in sorted(rows_of):
        rows = rows_of[e]
        ew = {kk: f64(v) for kk, v in expert_of(e).items() if v is not None}
        ts = [t for (t, _) in rows]
        xe = xs[ts]
        oe = O.expert_apply(activation, xe, ew)
        g = np.array([gate[t, k] for (t, k) in rows])
        for r, (t, k) in enumerate(rows):
            dg[t, k] = float(dys[t] @ oe[r])
        do = g[:, None] * dys[ts]
        bw = expert_backward(activation, xe, ew, do)
        if e in exps:
            dw[e] = {kk: v for kk, v in bw.items() if kk != "dx"}
        for r, t in enumerate(ts):
            if t in tok_set:
                dx_rows[t] = dx_rows.get(t, 0.0) + bw["dx"][r]
    # experts with no kept row: zero weight gradient
    for e in exps:
        if e < N and e not in dw:
            ew = {kk: f64(v) for kk, v in expert_of(e).items() if v is not None}
            dw[e] = {"d" + kk: np.zeros_like(v) for kk, v in ew.items()}
    # shared experts: every token, gate 1, do = dy
    for s in range(n_shared):
        e = N + s
        ew = {kk: f64(v) for kk, v in expert_of(e).items() if v is not None}
        if e in exps:
            bw = expert_backward(activation, xs, ew, dys)
            dw[e] = {kk: v for kk, v in bw.items() if kk != "dx"}
            dxs = bw["dx"][tok]
        else:
            dxs = expert_backward(activation, xs[tok], ew, dys[tok])["dx"]
        for i, t in enumerate(tok):
            dx_rows[int(t)] = dx_rows.get(int(t), 0.0) + dxs[i]

    dl = logit_grad(l, idx, gate, dg, f, alpha=alpha, z_coef=z_coef, gate_mode=gate_mode)
    wr = f64(w_r)
    dx = np.zeros((len(tok), d))
    for i, t in enumerate(tok):
        acc = dl[t] @ wr + (dys[t] if add_residual else 0.0)
        if int(t) in dx_rows:
            acc = acc + dx_rows[int(t)]
        dx[i] = acc
    out = {"dx": dx, "dw": dw, "tokens": tok, "fwd": fwd}
    if need_all_dg:
        out["dg"] = dg
        out["dl"] = dl
    if router_grads:
        out["dw_r"] = dl.T @ xs
        if b_r is not None:
            out["db_r"] = dl.sum(axis=0)
    return out


def objective(x, w_r, b_r, expert_of, dy, *, K: int, activation: str,
              capacity_factor: float = math.inf, alpha: float = 0.01, z_coef: float = 0.0,
              add_residual: bool = False, gate_mode: str = "renorm", select_bias=None,
              n_shared: int = 0, idx_override=None) -> float:
    """L = <dy, y> + L_aux + z_coef * z_loss, from the forward oracle."""
    fwd = O.moe_forward(x, w_r, b_r, expert_of, K=K, activation=activation,
                        capacity_factor=capacity_factor, alpha=alpha,
                        add_residual=add_residual, idx_override=idx_override,
                        gate_mode=gate_mode, select_bias=select_bias, n_shared=n_shared)
    return float(np.sum(f64(dy) * fwd["y"]) + fwd["l_aux"] + z_coef * fwd["z_loss"])
