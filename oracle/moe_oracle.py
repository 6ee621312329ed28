"""Float64 CPU oracle of the sparse Mixture-of-Experts forward layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
run this module: only the tests, the smoke check of the package entry file
and the CPU-baseline / reference legs of the benchmark script use it. It
shares no code with the CUDA path; both take their inputs from the seeded
generators in moe_inputs.py.

It is the plain definition of what the layer computes, written out step by
step in float64 (numpy; matrix products, sorts and erf are library calls):
every stored input (bf16 or fp32) is promoted exactly to float64 and nothing
is rounded on the way. Each function names the passage it follows. Sources:

  [MoE核心思想]  "MoE 的核心思想" (wmrh.cn): 公式表达重点, 具体数值示例,
                 专家容量, 辅助损失公式, Router Z-Loss.
  [稀疏激活原理] "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战"
                 (mzlw.cn): §2.1, §2.2, §2.3, §三 (Expert, MoERouter,
                 MoELayer).
  [概念卡]       "混合专家模型（Mixture of Experts, MoE）" (learnagent.wiki):
                 结构 2, 结构 3, 结构 4, 运行示例.
  [替代FFN]      "MoE 如何替代 FFN？它解决了什么问题？带来哪些新挑战？"
                 (mstx.cn): §1, §2, §4 (6), §5.

Readings where the pages are silent or disagree (each one is listed with its
reason in the design notes):
  * gates are renormalised over the K selected experts (softmax of the K
    selected logits), not the unrenormalised full softmax;
  * capacity C = floor(K * CF * T / N) with T = batch * seq_len, exact on
    the rational value of CF; CF <= 0 or CF = inf means no limit;
  * capacity is per expert over all ranks; assignments are visited rank-major
    (k ascending, then t ascending) and the first C of each expert are kept;
  * a dropped assignment contributes 0 and the surviving gates are not
    renormalised again; with the residual on, the token passes as x;
  * f_i counts assignments before capacity, over T*K;
  * ties in top-K go to the lower expert index; selection compares logits;
  * GELU is the exact-erf form;
  * router z-loss (no formula on the pages) is the mean over tokens of the
    squared log-sum-exp of the logits; the selection bias changes the top-K
    choice only;
  * shared experts (named, not formulated, on the pages) take every token
    with gate 1, bypass router and capacity and stay out of the statistics.

Every function here is pinned by tests/test_oracle_pins.py against values
the pages print, closed forms, special cases and brute force.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
from scipy.special import erf as _erf


# --------------------------------------------------------------------------
# conversions
# --------------------------------------------------------------------------
def f64(a) -> np.ndarray:
    """Exact promotion of a stored tensor (numpy, or torch incl. bf16) to float64."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return a.astype(np.float64, copy=False)
    # torch tensor: promote on the CPU (bf16 -> float64 is exact)
    return a.detach().to("cpu").double().numpy()


# --------------------------------------------------------------------------
# router: [稀疏激活原理] §2.1, §三 MoERouter.forward; [概念卡] 结构 2
# --------------------------------------------------------------------------
def router_logits(x, w_r, b_r=None) -> np.ndarray:
    """logits[t, e] = sum_j x[t, j] * W_r[e, j] (+ b_r[e]).

    [稀疏激活原理] §2.1: logits = x · W_r with W_r in R^{d x N}; the class
    MoERouter stores the weight as (N, d) and computes x @ W^T.
    [概念卡] 运行示例: the router is nn.Linear(hidden, N), i.e. with a bias."""
    x = f64(x)
    w = f64(w_r)
    l = x @ w.T
    if b_r is not None:
        l = l + f64(b_r)[None, :]
    return l


def softmax(l: np.ndarray) -> np.ndarray:
    """Row softmax, max-subtracted. [概念卡] 结构 2: G(x) = Softmax(W_r x)."""
    m = l.max(axis=-1, keepdims=True)
    z = np.exp(l - m)
    return z / z.sum(axis=-1, keepdims=True)


def topk_experts(l: np.ndarray, K: int) -> np.ndarray:
    """The K experts with the largest logits, in descending order of logit;
    equal logits rank the lower expert index first.

    [稀疏激活原理] §2.1 (Top-K 选择) and §三 (torch.topk(logits, top_k));
    the pages leave ties open, so the lower index wins (a stable sort)."""
    order = np.argsort(-l, axis=-1, kind="stable")
    return order[:, :K].astype(np.int64)


def renormalised_gates(l: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """g[t, k] = exp(l[t, idx_k]) / sum_k' exp(l[t, idx_k']).

    [稀疏激活原理] §三 MoERouter.forward: softmax over the top-K logits only;
    [MoE核心思想] 公式表达重点: G_i(x) are renormalised gate weights."""
    sel = np.take_along_axis(l, idx, axis=-1)
    m = sel.max(axis=-1, keepdims=True)
    z = np.exp(sel - m)
    return z / z.sum(axis=-1, keepdims=True)


# The pages state the gate in two more ways; the pins check all three agree.
def gates_softmax_then_topk(l: np.ndarray, K: int):
    """[概念卡] 运行示例: p = softmax(router(x)); (w, idx) = topk(p, K);
    w = w / sum(w). Returns (idx, w)."""
    p = softmax(l)
    idx = np.argsort(-p, axis=-1, kind="stable")[:, :K]
    w = np.take_along_axis(p, idx, axis=-1)
    return idx, w / w.sum(axis=-1, keepdims=True)


def gates_masked_softmax(l: np.ndarray, K: int):
    """[MoE核心思想] 公式表达重点: the scores outside the top K are set to -inf
    and the softmax is taken over all N; the top-K positions carry the
    gates. Returns (idx, g) with g read at idx."""
    idx = topk_experts(l, K)
    masked = np.full_like(l, -np.inf)
    np.put_along_axis(masked, idx, np.take_along_axis(l, idx, axis=-1), axis=-1)
    m = masked.max(axis=-1, keepdims=True)
    z = np.exp(masked - m)          # exp(-inf) = 0 outside the top K
    p = z / z.sum(axis=-1, keepdims=True)
    return idx, np.take_along_axis(p, idx, axis=-1)


# --------------------------------------------------------------------------
# gate variants (the further router options the pages name)
# --------------------------------------------------------------------------
def topk_with_selection_bias(l: np.ndarray, K: int, select_bias=None) -> np.ndarray:
    """[概念卡] 结构 4 (auxiliary-loss-free balancing, DeepSeek-V3): a per-expert
    bias, updated outside the gradient from how often each expert is chosen,
    steers which experts are selected. It enters the top-K choice only; the
    gates and the statistics use the unbiased logits. None = no bias."""
    if select_bias is None:
        return topk_experts(l, K)
    return topk_experts(l + f64(select_bias)[None, :], K)


def full_softmax_gates(l: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """[稀疏激活原理] §2.1 formula h(x) = Σ_{i∈TopK} softmax(logits)_i E_i(x):
    the selected experts' probabilities under the softmax over all N experts,
    not renormalised (the Switch-style gate; with K=1 it is the top
    probability)."""
    return np.take_along_axis(softmax(l), idx, axis=-1)


def router_z_loss(l: np.ndarray) -> float:
    """[MoE核心思想] Router Z-Loss: a penalty on the size of the router logits;
    the page gives no formula. Read as the ST-MoE form, the mean over tokens
    of (log Σ_e exp l[t, e])^2."""
    if l.shape[0] == 0:
        return 0.0
    m = l.max(axis=-1)
    lse = m + np.log(np.exp(l - m[:, None]).sum(axis=-1))
    return float(np.mean(lse ** 2))


def routing_entropy(p: np.ndarray) -> float:
    """[替代FFN] §4 (6) monitors the routing entropy: the mean over tokens of
    -Σ_e p[t, e] log p[t, e] (0 log 0 = 0)."""
    if p.shape[0] == 0:
        return 0.0
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(p > 0, p * np.log(p), 0.0)
    return float(np.mean(-t.sum(axis=-1)))


# --------------------------------------------------------------------------
# load-balance statistics: [稀疏激活原理] §2.2 and §三
# _compute_load_balance_loss; [MoE核心思想] 辅助损失公式
# --------------------------------------------------------------------------
def load_balance(idx: np.ndarray, p: np.ndarray, N: int, alpha: float):
    """count[e] = #{(t, k): idx[t, k] = e}; f = count / (T*K);
    P = mean over tokens of the router softmax; L_aux = alpha * N * sum f*P.
    f is taken before capacity (the page computes it from the top-k indices)."""
    T, K = idx.shape
    count = np.bincount(idx.reshape(-1), minlength=N).astype(np.int64)
    f = count / float(T * K) if T > 0 else np.zeros(N)
    P = p.mean(axis=0) if T > 0 else np.zeros(N)
    l_aux = float(alpha) * N * float(np.sum(f * P))
    return count, f, P, l_aux


# --------------------------------------------------------------------------
# capacity and dispatch: [稀疏激活原理] §2.3, §三 MoELayer.forward;
# [MoE核心思想] 专家容量
# --------------------------------------------------------------------------
def capacity(K: int, N: int, capacity_factor: float, T: int):
    """C = floor(K/N * CF * T) on the exact rational value of CF.
    Returns None (no limit) when CF <= 0 or CF is infinite."""
    cf = float(capacity_factor)
    if math.isnan(cf):
        raise ValueError("capacity factor is NaN")
    if cf <= 0 or math.isinf(cf):
        return None
    return math.floor(Fraction(K) * Fraction(cf) * Fraction(T) / Fraction(N))


def dispatch(idx: np.ndarray, N: int, C):
    """Visit the assignments rank-major (k = 0..K-1, then t ascending); an
    assignment to expert e is kept while expert e has taken fewer than C.
    Kept assignments of expert e take consecutive slots from offsets[e] in
    visiting order. Returns a dict with count, kept, offsets (N+1), slot_of
    [T][K] (-1 if dropped), token_of_slot [A], rank_of [T][K] (-1 if
    dropped) and n_dropped."""
    T, K = idx.shape
    limit = math.inf if C is None else C
    filled = np.zeros(N, dtype=np.int64)
    rank_of = np.full((T, K), -1, dtype=np.int64)
    count = np.zeros(N, dtype=np.int64)
    for k in range(K):
        for t in range(T):
            e = int(idx[t, k])
            count[e] += 1
            if filled[e] < limit:
                rank_of[t, k] = filled[e]
                filled[e] += 1
    offsets = np.zeros(N + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(filled)
    slot_of = np.full((T, K), -1, dtype=np.int64)
    token_of_slot = np.zeros(int(offsets[N]), dtype=np.int64)
    for k in range(K):
        for t in range(T):
            r = rank_of[t, k]
            if r >= 0:
                s = offsets[idx[t, k]] + r
                slot_of[t, k] = s
                token_of_slot[s] = t
    return {"count": count, "kept": filled, "offsets": offsets, "slot_of": slot_of,
            "token_of_slot": token_of_slot, "rank_of": rank_of,
            "n_dropped": int(count.sum() - filled.sum())}


# --------------------------------------------------------------------------
# experts: [稀疏激活原理] §三 class Expert (SwiGLU); [概念卡] 运行示例 (GELU);
# [替代FFN] §1 (FFN(x) = W_2 act(W_1 x))
# --------------------------------------------------------------------------
def silu(a: np.ndarray) -> np.ndarray:
    """silu(a) = a * sigmoid(a) = a / (1 + e^-a)."""
    return a / (1.0 + np.exp(-a))


def gelu_erf(z: np.ndarray) -> np.ndarray:
    """Exact GELU (nn.GELU's default): z/2 * (1 + erf(z / sqrt 2))."""
    return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))


def expert_swiglu(xe, w_gate, w_up, w_down) -> np.ndarray:
    """down(silu(gate(x)) * up(x)) without biases (the SwiGLU workloads)."""
    xe = f64(xe)
    h = silu(xe @ f64(w_gate).T) * (xe @ f64(w_up).T)
    return h @ f64(w_down).T


def expert_gelu(xe, w1, b1, w2, b2) -> np.ndarray:
    """Linear(d -> F) -> GELU -> Linear(F -> d); biases optional."""
    xe = f64(xe)
    z = xe @ f64(w1).T
    if b1 is not None:
        z = z + f64(b1)[None, :]
    o = gelu_erf(z) @ f64(w2).T
    if b2 is not None:
        o = o + f64(b2)[None, :]
    return o


def expert_apply(activation: str, xe, ew: dict) -> np.ndarray:
    """Apply one expert; ew holds that expert's weights."""
    if activation == "swiglu":
        return expert_swiglu(xe, ew["w_gate"], ew["w_up"], ew["w_down"])
    return expert_gelu(xe, ew["w1"], ew.get("b1"), ew["w2"], ew.get("b2"))


def stacked_expert(weights: dict, e: int) -> dict:
    """Slice expert e out of stacked [N][...] weights (numpy or torch)."""
    return {k: v[e] for k, v in weights.items() if v is not None}


# --------------------------------------------------------------------------
# the layer: [稀疏激活原理] §三 MoELayer.forward; [概念卡] 核心原理 (four
# steps) and 结构 3 (y = Σ_{i∈TopK} G(x)_i E_i(x))
# --------------------------------------------------------------------------
def shared_experts_output(xs: np.ndarray, expert_of, N: int, n_shared: int,
                          activation: str) -> np.ndarray:
    """[替代FFN] §5 (DeepSeek-MoE: fine-grained experts plus shared experts):
    the shared experts N .. N+n_shared-1 run on every token with gate 1,
    outside the router and the capacity, and their outputs add to the layer
    output."""
    out = np.zeros_like(xs)
    for s in range(n_shared):
        ew = {kk: f64(v) for kk, v in expert_of(N + s).items() if v is not None}
        out = out + expert_apply(activation, xs, ew)
    return out


def moe_forward(x, w_r, b_r, expert_of, *, K: int, activation: str,
                capacity_factor: float = math.inf, alpha: float = 0.01,
                add_residual: bool = False, tokens=None, idx_override=None,
                gate_mode: str = "renorm", select_bias=None, n_shared: int = 0):
    """The whole layer in float64.

    expert_of(e) returns expert e's weights (dict of arrays, promoted here).
    tokens: evaluate y only for these token indices (routing, statistics and
    dispatch always cover all tokens); None = all tokens.
    idx_override: use this routing instead of the oracle's top-K (to follow a
    GPU choice among near-tied logits); gates are recomputed from it.
    gate_mode: "renorm" (softmax over the K selected logits) or "softmax"
    (full-softmax probabilities, not renormalised). select_bias: [N] bias
    for the top-K choice only. n_shared: shared experts (indices N.. of
    expert_of) added to every token with gate 1.
    Returns a dict of every intermediate the layer defines."""
    xs = f64(x)
    T = xs.shape[0]
    l = router_logits(xs, w_r, b_r)
    N = l.shape[1]
    p = softmax(l) if T > 0 else np.zeros((0, N))
    idx = (topk_with_selection_bias(l, K, select_bias) if idx_override is None
           else np.asarray(idx_override, dtype=np.int64))
    if T == 0:
        gate = np.zeros((0, K))
    elif gate_mode == "renorm":
        gate = renormalised_gates(l, idx)
    else:
        gate = full_softmax_gates(l, idx)
    count, f, P, l_aux = load_balance(idx, p, N, alpha)
    C = capacity(K, N, capacity_factor, T)
    disp = dispatch(idx, N, C)

    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    y = np.zeros((len(tok), xs.shape[1]))
    # group the kept assignments of the requested tokens by expert
    by_expert = {}
    for i, t in enumerate(tok):
        for k in range(K):
            if disp["slot_of"][t, k] >= 0:
                by_expert.setdefault(int(idx[t, k]), []).append((i, int(t), k))
    o_of = {}
    for e in sorted(by_expert):
        rows = by_expert[e]
        ew = {kk: f64(v) for kk, v in expert_of(e).items() if v is not None}
        oe = expert_apply(activation, xs[[t for (_, t, _) in rows]], ew)
        for r, (i, t, k) in enumerate(rows):
            o_of[(i, k)] = oe[r]
    shared = (shared_experts_output(xs[tok], expert_of, N, n_shared, activation)
              if n_shared > 0 and len(tok) > 0 else None)
    for i, t in enumerate(tok):
        acc = np.zeros(xs.shape[1])
        for k in range(K):
            if (i, k) in o_of:
                acc = acc + gate[t, k] * o_of[(i, k)]
        if shared is not None:
            acc = acc + shared[i]
        y[i] = acc + (xs[t] if add_residual else 0.0)
    return {"logits": l, "p": p, "idx": idx, "gate": gate, "count": count, "f": f,
            "P": P, "l_aux": l_aux, "z_loss": router_z_loss(l), "entropy": routing_entropy(p),
            "C": C, "tokens": tok, "y": y, **{
                k: disp[k] for k in ("kept", "offsets", "slot_of", "token_of_slot",
                                     "rank_of", "n_dropped")}}


def dense_all_experts(x, w_r, b_r, expert_of, *, K: int, activation: str) -> np.ndarray:
    """[概念卡] 运行示例: evaluate every expert on every token, then gather the
    top-K outputs and weight them (softmax -> top-K -> renormalise). No
    capacity. Brute force for tiny inputs."""
    xs = f64(x)
    l = router_logits(xs, w_r, b_r)
    idx, w = gates_softmax_then_topk(l, K)
    N = l.shape[1]
    all_out = np.stack([expert_apply(activation, xs,
                                     {kk: f64(v) for kk, v in expert_of(e).items()
                                      if v is not None})
                        for e in range(N)], axis=1)          # [T][N][d]
    out = np.zeros_like(xs)
    for k in range(K):
        out += w[:, k:k + 1] * np.take_along_axis(all_out, idx[:, k][:, None, None],
                                                  axis=1)[:, 0, :]
    return out


# --------------------------------------------------------------------------
# near-ties: the routing of a token whose sorted top-(K+1) logits have an
# adjacent gap below eps depends on rounding; such tokens are reported apart
# --------------------------------------------------------------------------
def near_tie_tokens(l: np.ndarray, K: int, eps: float = 1e-5) -> np.ndarray:
    """Boolean [T]: some adjacent gap among the K+1 largest logits is < eps
    (among the K largest when K = N)."""
    srt = -np.sort(-l, axis=-1)
    m = min(K + 1, l.shape[1])
    if m < 2:
        return np.zeros(l.shape[0], dtype=bool)
    gaps = srt[:, :m - 1] - srt[:, 1:m]
    return (gaps < eps).any(axis=-1)
