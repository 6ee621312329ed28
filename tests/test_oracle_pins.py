"""Pins of the float64 oracle against what the pages and mathematics fix.

Each test ties one oracle function to something other than itself: a value
the pages print (tests/golden/), a closed form, an identity between two of
the pages' own formulations, a special case that reduces to a library
routine, or brute force on tiny inputs. The mutation tests at the end plant
plausible mistakes in the oracle (on the CPU) and check that a pin catches
each of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- gates ----
def check_worked_example(golden):
    kv, _ = golden("worked_example_topk2.txt")
    l = np.array([kv["logits"]])
    K = int(kv["top_k"][0])
    idx = O.topk_experts(l, K)
    g = O.renormalised_gates(l, idx)
    assert list(idx[0]) == [int(v) for v in kv["expected_experts"]]
    assert [round(float(v), 2) for v in g[0]] == kv["expected_gates_2dp"]
    assert abs(g[0, 0] - 2.0 / 3.0) < 1e-15 and abs(g[0, 1] - 1.0 / 3.0) < 1e-15


def test_worked_example_gates(golden):
    """"MoE 的核心思想", 具体数值示例: experts 6 and 2 with 0.67 / 0.33."""
    check_worked_example(golden)


def test_worked_example_other_formulations(golden):
    kv, _ = golden("worked_example_topk2.txt")
    l = np.array([kv["logits"]])
    for fn in (O.gates_softmax_then_topk, O.gates_masked_softmax):
        idx, g = fn(l, 2)
        assert list(idx[0]) == [6, 2]
        assert [round(float(v), 2) for v in g[0]] == [0.67, 0.33]


@pytest.mark.parametrize("N,K", [(4, 1), (4, 2), (8, 2), (64, 1), (64, 4), (256, 8), (5, 5)])
def test_three_gate_formulations_agree(N, K):
    """Top-K then softmax (mzlw §三), softmax then top-K then renormalise
    (learnagent 运行示例) and the -inf mask then softmax (wmrh 公式表达重点)
    are the same gate."""
    rng = np.random.default_rng(N * 31 + K)
    l = rng.normal(0, 2.0, size=(500, N))
    idx = O.topk_experts(l, K)
    g = O.renormalised_gates(l, idx)
    idx2, g2 = O.gates_softmax_then_topk(l, K)
    idx3, g3 = O.gates_masked_softmax(l, K)
    assert np.array_equal(idx, idx2) and np.array_equal(idx, idx3)
    assert np.max(np.abs(g - g2)) < 1e-14 and np.max(np.abs(g - g3)) < 1e-14
    assert np.allclose(g.sum(-1), 1.0, atol=1e-14, rtol=0)
    assert (np.diff(np.take_along_axis(l, idx, -1), axis=-1) <= 0).all()  # descending


def test_topk_ties_lower_index_and_bruteforce():
    rng = np.random.default_rng(7)
    l = rng.integers(0, 3, size=(200, 6)).astype(np.float64)  # many exact ties
    for K in range(1, 7):
        idx = O.topk_experts(l, K)
        for t in range(l.shape[0]):
            ref = sorted(range(6), key=lambda e: (-l[t, e], e))[:K]
            assert list(idx[t]) == ref


def test_softmax_closed_forms():
    assert np.allclose(O.softmax(np.zeros((1, 8))), 1.0 / 8, atol=1e-16, rtol=0)
    p = O.softmax(np.array([[0.0, math.log(2.0)]]))
    assert abs(p[0, 0] - 1 / 3) < 1e-15 and abs(p[0, 1] - 2 / 3) < 1e-15
    # shift invariance and a library routine
    rng = np.random.default_rng(3)
    l = rng.normal(size=(50, 17)) * 10
    ref = torch.softmax(torch.from_numpy(l), dim=-1).numpy()
    assert np.max(np.abs(O.softmax(l) - ref)) < 1e-15
    assert np.max(np.abs(O.softmax(l + 123.0) - O.softmax(l))) < 1e-14


def test_router_logits_library_and_bias():
    rng = np.random.default_rng(11)
    x = rng.normal(size=(9, 13))
    w = rng.normal(size=(5, 13))
    b = rng.normal(size=5)
    l = O.router_logits(x, w, b)
    # brute force double loop
    for t in range(9):
        for e in range(5):
            assert abs(l[t, e] - (sum(x[t, j] * w[e, j] for j in range(13)) + b[e])) < 1e-12
    # nn.Linear in float64 is the page's router (learnagent 运行示例)
    lin = torch.nn.Linear(13, 5, dtype=torch.float64)
    with torch.no_grad():
        lin.weight.copy_(torch.from_numpy(w))
        lin.bias.copy_(torch.from_numpy(b))
        ref = lin(torch.from_numpy(x)).numpy()
    assert np.max(np.abs(l - ref)) < 1e-13


# ------------------------------------------------------ load balancing ----
def test_laux_balanced_is_alpha():
    """mzlw §2.2: f_i = p_i = 1/N gives L_aux = alpha. Rotating one logit
    vector through all N positions makes both exactly uniform."""
    for N, K in [(4, 2), (8, 2), (64, 1), (256, 8)]:
        rng = np.random.default_rng(N)
        base = rng.normal(size=N)
        l = np.stack([np.roll(base, t) for t in range(3 * N)])
        idx = O.topk_experts(l, K)
        count, f, P, laux = O.load_balance(idx, O.softmax(l), N, 0.01)
        assert np.all(count == 3 * K)
        assert np.max(np.abs(P - 1.0 / N)) < 1e-15
        assert abs(laux - 0.01) < 1e-15


def test_laux_collapsed_split(golden):
    """mzlw §2.2 figure 坍缩路由: 70/20/8/2 over 4 experts, f = P."""
    kv, _ = golden("laux_collapse.txt")
    alpha = kv["alpha"][0]
    split = kv["collapsed_split"]
    T = 100
    idx = np.concatenate([np.full(int(round(s * T)), e) for e, s in enumerate(split)])[:, None]
    l = np.full((T, 4), -1000.0)
    l[np.arange(T), idx[:, 0]] = 0.0          # one-hot softmax rows: P = f exactly
    count, f, P, laux = O.load_balance(idx, O.softmax(l), 4, alpha)
    assert np.allclose(f, split, atol=1e-15, rtol=0) and np.allclose(P, split, atol=1e-15, rtol=0)
    assert abs(laux - kv["expected_laux_collapsed"][0]) < 1e-15
    assert laux > kv["expected_laux_balanced"][0]


def test_laux_cauchy_schwarz_when_f_equals_P():
    rng = np.random.default_rng(5)
    for _ in range(50):
        N = int(rng.integers(2, 40))
        f = rng.dirichlet(np.ones(N))
        assert N * np.sum(f * f) >= 1 - 1e-15


def test_count_f_definition():
    rng = np.random.default_rng(9)
    T, N, K = 40, 6, 3
    l = rng.normal(size=(T, N))
    idx = O.topk_experts(l, K)
    count, f, P, _ = O.load_balance(idx, O.softmax(l), N, 0.01)
    for e in range(N):
        assert count[e] == sum(1 for t in range(T) for k in range(K) if idx[t, k] == e)
    assert abs(f.sum() - 1.0) < 1e-15 and abs(P.sum() - 1.0) < 1e-14


# ------------------------------------------------------------ capacity ----
def test_capacity_golden(golden):
    _, rows = golden("capacity_cases.txt")
    for K, N, cf, T, C in rows:
        assert O.capacity(int(K), int(N), cf, int(T)) == int(C)


def test_capacity_is_floor_and_unlimited_cases():
    from fractions import Fraction
    assert O.capacity(2, 8, math.inf, 100) is None
    assert O.capacity(2, 8, 0.0, 100) is None
    assert O.capacity(2, 8, -1.0, 100) is None
    for K, N, T in itertools.product([1, 2, 3, 8], [1, 3, 8, 64], [1, 7, 100, 4096]):
        for cf32 in np.float32([0.1, 0.7, 1.0, 1.25, 1.3333, 2.5]):
            cf = float(cf32)
            C = O.capacity(K, N, cf, T)
            exact = Fraction(K) * Fraction(cf) * Fraction(T) / Fraction(N)
            assert C <= exact < C + 1


# ------------------------------------------------------------ dispatch ----
def brute_force_dispatch(idx, N, C):
    """Per expert: sort its assignments by (k, t); the first C are kept."""
    T, K = idx.shape
    kept_lists = []
    for e in range(N):
        asg = sorted((k, t) for t in range(T) for k in range(K) if idx[t, k] == e)
        kept_lists.append(asg if C is None else asg[:C])
    slot_of = -np.ones((T, K), dtype=np.int64)
    base = 0
    for e in range(N):
        for r, (k, t) in enumerate(kept_lists[e]):
            slot_of[t, k] = base + r
        base += len(kept_lists[e])
    return slot_of, [len(v) for v in kept_lists]


@pytest.mark.parametrize("T,N,K,C", [(50, 4, 2, 10), (64, 8, 1, 3), (33, 5, 3, None),
                                     (100, 6, 2, 0), (17, 2, 2, 100), (1, 1, 1, 1)])
def test_dispatch_brute_force_and_invariants(T, N, K, C):
    rng = np.random.default_rng(T * N + K)
    l = rng.normal(size=(T, N)) + np.linspace(2, 0, N)  # skewed towards low experts
    idx = O.topk_experts(l, K)
    d = O.dispatch(idx, N, C)
    slot_bf, kept_bf = brute_force_dispatch(idx, N, C)
    assert np.array_equal(d["slot_of"], slot_bf)
    assert list(d["kept"]) == kept_bf
    count = np.bincount(idx.reshape(-1), minlength=N)
    cap = np.inf if C is None else C
    assert list(d["kept"]) == [int(min(c, cap)) for c in count]
    assert d["n_dropped"] == int(sum(max(0, c - cap) for c in count))
    assert d["n_dropped"] == int((d["slot_of"] < 0).sum())
    assert list(d["offsets"]) == [0] + list(np.cumsum(d["kept"]))
    for t in range(T):
        for k in range(K):
            s = d["slot_of"][t, k]
            if s >= 0:
                assert d["token_of_slot"][s] == t
                assert d["offsets"][idx[t, k]] <= s < d["offsets"][idx[t, k] + 1]


def test_switch_capacity_drop_count():
    """K=1, CF=1.25: the drop count equals sum_e max(0, count_e - C)."""
    rng = np.random.default_rng(2)
    T, N = 2048, 64
    l = rng.normal(size=(T, N))
    l[:, :4] += 1.5
    idx = O.topk_experts(l, 1)
    C = O.capacity(1, N, 1.25, T)
    assert C == 40
    d = O.dispatch(idx, N, C)
    count = np.bincount(idx[:, 0], minlength=N)
    assert d["n_dropped"] == int(np.maximum(count - C, 0).sum()) > 0


# ------------------------------------------------------------- experts ----
def test_activations_against_library_and_identities():
    z = np.linspace(-12, 12, 2001)
    tz = torch.from_numpy(z)
    assert np.max(np.abs(O.gelu_erf(z) - torch.nn.functional.gelu(tz).numpy())) < 1e-14
    assert np.max(np.abs(O.silu(z) - torch.nn.functional.silu(tz).numpy())) < 1e-14
    assert np.max(np.abs(O.gelu_erf(z) - O.gelu_erf(-z) - z)) < 1e-13
    assert np.max(np.abs(O.silu(z) - O.silu(-z) - z)) < 1e-13
    assert O.gelu_erf(np.array([0.0]))[0] == 0.0 and O.silu(np.array([0.0]))[0] == 0.0


def test_experts_against_torch_modules():
    """mzlw §三 class Expert (SwiGLU) and learnagent 运行示例 (GELU) as
    nn.Linear stacks in float64."""
    rng = np.random.default_rng(4)
    d, F, M = 12, 20, 7
    x = torch.from_numpy(rng.normal(size=(M, d)))
    gate = torch.nn.Linear(d, F, bias=False, dtype=torch.float64)
    up = torch.nn.Linear(d, F, bias=False, dtype=torch.float64)
    down = torch.nn.Linear(F, d, bias=False, dtype=torch.float64)
    with torch.no_grad():
        ref = down(torch.nn.functional.silu(gate(x)) * up(x)).numpy()
    got = O.expert_swiglu(x, gate.weight, up.weight, down.weight)
    assert np.max(np.abs(got - ref)) < 1e-13
    seq = torch.nn.Sequential(torch.nn.Linear(d, F, dtype=torch.float64), torch.nn.GELU(),
                              torch.nn.Linear(F, d, dtype=torch.float64))
    with torch.no_grad():
        ref = seq(x).numpy()
    got = O.expert_gelu(x, seq[0].weight, seq[0].bias, seq[2].weight, seq[2].bias)
    assert np.max(np.abs(got - ref)) < 1e-13


# ------------------------------------------------------- whole layer ----
def tiny_layer(activation, T=10, d=8, F=12, N=4, seed=0, bias=True):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, d))
    w_r = rng.normal(size=(N, d))
    b_r = rng.normal(size=N) if bias else None
    if activation == "swiglu":
        W = {"w_gate": rng.normal(size=(N, F, d)) * 0.3, "w_up": rng.normal(size=(N, F, d)) * 0.3,
             "w_down": rng.normal(size=(N, d, F)) * 0.3}
    else:
        W = {"w1": rng.normal(size=(N, F, d)) * 0.3, "b1": rng.normal(size=(N, F)) * 0.1,
             "w2": rng.normal(size=(N, d, F)) * 0.3, "b2": rng.normal(size=(N, d)) * 0.1}
    return x, w_r, b_r, W, (lambda e: O.stacked_expert(W, e))


@pytest.mark.parametrize("activation", ["swiglu", "gelu"])
@pytest.mark.parametrize("K", [1, 2, 3])
def test_sparse_equals_dense_brute_force(activation, K):
    """learnagent 运行示例 evaluates all experts then gathers: same result."""
    x, w_r, b_r, W, ex = tiny_layer(activation)
    r = O.moe_forward(x, w_r, b_r, ex, K=K, activation=activation)
    dense = O.dense_all_experts(x, w_r, b_r, ex, K=K, activation=activation)
    assert np.max(np.abs(r["y"] - dense)) < 1e-12


def test_single_expert_is_plain_ffn():
    """mstx §1: with N = K = 1 the layer is the dense FFN W_2 act(W_1 x)."""
    x, w_r, b_r, W, ex = tiny_layer("gelu", N=1)
    r = O.moe_forward(x, w_r, b_r, ex, K=1, activation="gelu")
    z = x @ W["w1"][0].T + W["b1"][0]
    ffn = (0.5 * z * (1 + torch.erf(torch.from_numpy(z) / math.sqrt(2)).numpy())) @ W["w2"][0].T \
        + W["b2"][0]
    assert np.max(np.abs(r["y"] - ffn)) < 1e-12
    assert np.all(r["gate"] == 1.0)


def test_k_equals_n_is_dense_softmax_mixture():
    x, w_r, b_r, W, ex = tiny_layer("swiglu", N=5)
    r = O.moe_forward(x, w_r, b_r, ex, K=5, activation="swiglu")
    p = torch.softmax(torch.from_numpy(x @ w_r.T + b_r), -1).numpy()
    outs = [O.expert_swiglu(x, W["w_gate"][e], W["w_up"][e], W["w_down"][e]) for e in range(5)]
    mix = sum(p[:, e:e + 1] * outs[e] for e in range(5))
    assert np.max(np.abs(r["y"] - mix)) < 1e-12


def test_top1_is_argmax_expert():
    x, w_r, b_r, W, ex = tiny_layer("swiglu", N=6)
    r = O.moe_forward(x, w_r, b_r, ex, K=1, activation="swiglu")
    am = np.argmax(x @ w_r.T + b_r, axis=-1)
    for t in range(x.shape[0]):
        e = am[t]
        ref = O.expert_swiglu(x[t:t + 1], W["w_gate"][e], W["w_up"][e], W["w_down"][e])[0]
        assert np.max(np.abs(r["y"][t] - ref)) < 1e-12


@pytest.mark.parametrize("residual", [False, True])
def test_zero_capacity_passes_tokens_through(residual):
    """mzlw §2.3: dropped tokens skip the experts and pass on the residual."""
    x, w_r, b_r, W, ex = tiny_layer("swiglu", T=6, N=8)
    r = O.moe_forward(x, w_r, b_r, ex, K=2, activation="swiglu", capacity_factor=0.01,
                      add_residual=residual)
    assert r["C"] == 0 and r["n_dropped"] == 12
    assert np.array_equal(r["y"], x if residual else np.zeros_like(x))


def test_partial_drop_no_renormalisation():
    """A token losing one of its two experts keeps the other expert's gate as is."""
    x, w_r, b_r, W, ex = tiny_layer("swiglu", T=20, N=4, seed=3)
    r = O.moe_forward(x, w_r, b_r, ex, K=2, activation="swiglu", capacity_factor=0.5)
    C = r["C"]
    assert C == 5
    hit = False
    for t in range(20):
        kept = [k for k in range(2) if r["slot_of"][t, k] >= 0]
        if len(kept) == 1:
            k = kept[0]
            e = r["idx"][t, k]
            ref = r["gate"][t, k] * O.expert_swiglu(x[t:t + 1], W["w_gate"][e], W["w_up"][e],
                                                    W["w_down"][e])[0]
            assert np.max(np.abs(r["y"][t] - ref)) < 1e-12
            hit = True
    assert hit


def test_token_subset_matches_full():
    x, w_r, b_r, W, ex = tiny_layer("gelu", T=30, N=4)
    full = O.moe_forward(x, w_r, b_r, ex, K=2, activation="gelu")
    sub = O.moe_forward(x, w_r, b_r, ex, K=2, activation="gelu", tokens=[3, 17, 29])
    assert np.max(np.abs(sub["y"] - full["y"][[3, 17, 29]])) < 1e-13


def test_near_tie_detection():
    l = np.array([[3.0, 3.0 - 5e-6, 1.0, 0.0],      # rank 0/1 gap below 1e-5
                  [3.0, 2.0, 2.0 - 2e-6, 0.0],      # rank 1/2 (K/K+1) gap below 1e-5
                  [3.0, 2.0, 1.0, 1.0 - 1e-7],      # only the rank 2/3 gap is small
                  [3.0, 2.0 + 2e-5, 2.0, 0.0]])     # all gaps >= 1e-5
    assert list(O.near_tie_tokens(l, 2)) == [True, True, False, False]


# ------------------------------------------- mutations caught by pins ----
def test_mutation_full_softmax_gate_is_caught(golden, monkeypatch):
    def wrong(l, idx):  # unrenormalised gate: read the full softmax at idx
        return np.take_along_axis(O.softmax(l), idx, axis=-1)
    monkeypatch.setattr(O, "renormalised_gates", wrong)
    with pytest.raises(AssertionError):
        check_worked_example(golden)


def test_mutation_token_major_dispatch_is_caught(monkeypatch):
    def wrong(idx, N, C):  # visits t outer, k inner: a different drop priority
        T, K = idx.shape
        limit = np.inf if C is None else C
        filled = np.zeros(N, dtype=np.int64)
        rank_of = -np.ones((T, K), dtype=np.int64)
        count = np.bincount(idx.reshape(-1), minlength=N)
        for t in range(T):
            for k in range(K):
                e = idx[t, k]
                if filled[e] < limit:
                    rank_of[t, k] = filled[e]
                    filled[e] += 1
        offsets = np.concatenate([[0], np.cumsum(filled)])
        slot_of = np.where(rank_of >= 0, offsets[idx] + rank_of, -1)
        tos = np.zeros(int(offsets[-1]), dtype=np.int64)
        for t in range(T):
            for k in range(K):
                if slot_of[t, k] >= 0:
                    tos[slot_of[t, k]] = t
        return {"count": count, "kept": filled, "offsets": offsets, "slot_of": slot_of,
                "token_of_slot": tos, "rank_of": rank_of,
                "n_dropped": int(count.sum() - filled.sum())}
    monkeypatch.setattr(O, "dispatch", wrong)
    with pytest.raises(AssertionError):
        test_dispatch_brute_force_and_invariants(50, 4, 2, 10)


def test_mutation_silu_sign_is_caught(monkeypatch):
    monkeypatch.setattr(O, "silu", lambda a: a / (1.0 + np.exp(a)))
    with pytest.raises(AssertionError):
        test_experts_against_torch_modules()


def test_mutation_gate_up_swapped_is_caught(monkeypatch):
    orig = O.expert_swiglu
    monkeypatch.setattr(O, "expert_swiglu",
                        lambda xe, w_gate, w_up, w_down: orig(xe, w_up, w_gate, w_down))
    with pytest.raises(AssertionError):
        test_experts_against_torch_modules()


def test_mutation_missing_router_bias_is_caught(monkeypatch):
    monkeypatch.setattr(O, "router_logits",
                        lambda x, w_r, b_r=None: O.f64(x) @ O.f64(w_r).T)
    with pytest.raises(AssertionError):
        test_router_logits_library_and_bias()


def test_mutation_f_after_capacity_is_caught(monkeypatch):
    def wrong(idx, p, N, alpha):  # counts only the first C=1 per expert
        count, f, P, laux = orig(idx[:1], p, N, alpha)
        return count, f, P, laux
    orig = O.load_balance
    monkeypatch.setattr(O, "load_balance", wrong)
    with pytest.raises(AssertionError):
        test_laux_balanced_is_alpha()


def test_switch_skew_bias_gives_seventy_percent():
    """The stored router bias of the skewed workload puts 70% +- 0.5% of the
    argmaxes on experts 0..3 (checked with the oracle's router)."""
    import moe_inputs
    w = moe_inputs.workload("switch_skewed")
    x = moe_inputs.make_x(w)
    w_r, b_r = moe_inputs.make_router(w)
    idx = O.topk_experts(O.router_logits(x, w_r, b_r), 1)
    share = float(np.mean(idx[:, 0] < moe_inputs.SWITCH_SKEW_EXPERTS))
    assert abs(share - 0.70) <= 0.005
    C = O.capacity(1, w.N, w.capacity_factor, w.T)
    assert C == 640


# ------------------------------------------------------ gate variants ----
def test_selection_bias_constant_shift_changes_nothing():
    rng = np.random.default_rng(21)
    l = rng.normal(size=(300, 16))
    for K in (1, 2, 5):
        a = O.topk_experts(l, K)
        b = O.topk_with_selection_bias(l, K, np.full(16, 3.7))
        assert np.array_equal(a, b)


def test_selection_bias_forces_expert_but_gate_uses_unbiased_logits():
    """[概念卡] 结构 4: a large bias on expert 3 puts it first in every top-2;
    its renormalised gate is still exp(l3) / (exp(l3) + exp(l_other))."""
    rng = np.random.default_rng(22)
    x = rng.normal(size=(40, 6))
    w_r = rng.normal(size=(5, 6))
    bias = np.zeros(5)
    bias[3] = 100.0
    W = {"w_gate": rng.normal(size=(5, 7, 6)), "w_up": rng.normal(size=(5, 7, 6)),
         "w_down": rng.normal(size=(5, 6, 7))}
    r = O.moe_forward(x, w_r, None, lambda e: O.stacked_expert(W, e), K=2, activation="swiglu",
                      select_bias=bias)
    l = x @ w_r.T
    assert np.all(r["idx"][:, 0] == 3)
    other = r["idx"][:, 1]
    lo = l[np.arange(40), other]
    expect = np.exp(l[:, 3]) / (np.exp(l[:, 3]) + np.exp(lo))
    assert np.max(np.abs(r["gate"][:, 0] - expect)) < 1e-14
    # statistics ignore the bias: P is the mean unbiased softmax
    assert np.max(np.abs(r["P"] - torch.softmax(torch.from_numpy(l), -1).numpy().mean(0))) < 1e-15


def test_full_softmax_gates_closed_forms():
    """[稀疏激活原理] §2.1 formula: g_i = softmax(logits)_i over all N."""
    l = np.array([[0.0, math.log(2.0), math.log(3.0), -np.inf]])
    idx = O.topk_experts(l, 2)
    g = O.full_softmax_gates(l, idx)
    assert list(idx[0]) == [2, 1]
    assert np.allclose(g[0], [3 / 6, 2 / 6], atol=1e-15, rtol=0)
    rng = np.random.default_rng(23)
    l = rng.normal(size=(100, 7))
    assert np.allclose(O.full_softmax_gates(l, O.topk_experts(l, 7)).sum(-1), 1.0, atol=1e-14)
    top1 = O.full_softmax_gates(l, O.topk_experts(l, 1))[:, 0]
    assert np.max(np.abs(top1 - O.softmax(l).max(-1))) < 1e-15


def test_z_loss_closed_forms():
    """Mean squared log-sum-exp: logits all c over N experts give (c + ln N)^2."""
    for N, c in [(4, 0.0), (8, 1.5), (64, -2.0)]:
        l = np.full((10, N), c)
        assert abs(O.router_z_loss(l) - (c + math.log(N)) ** 2) < 1e-12
    l = np.array([[1000.0, 0.0, 0.0]])  # one dominant logit: lse -> 1000
    assert abs(O.router_z_loss(l) - 1000.0 ** 2) < 1e-6
    rng = np.random.default_rng(24)
    l = rng.normal(size=(50, 9)) * 3
    ref = torch.logsumexp(torch.from_numpy(l), -1).numpy()
    assert abs(O.router_z_loss(l) - float(np.mean(ref ** 2))) < 1e-12


def test_routing_entropy_closed_forms():
    assert abs(O.routing_entropy(O.softmax(np.zeros((5, 8)))) - math.log(8)) < 1e-15
    assert O.routing_entropy(O.softmax(np.array([[0.0, -1e4, -1e4]]))) == 0.0
    two = O.softmax(np.array([[2.0, 2.0, -np.inf, -np.inf]]))
    assert abs(O.routing_entropy(two) - math.log(2)) < 1e-15


def test_mutation_biased_gate_is_caught(monkeypatch):
    orig = O.renormalised_gates
    def wrong(l, idx):  # gates computed on the biased logits
        return orig(l + np.eye(l.shape[1])[3] * 100.0, idx)
    monkeypatch.setattr(O, "renormalised_gates", wrong)
    with pytest.raises(AssertionError):
        test_selection_bias_forces_expert_but_gate_uses_unbiased_logits()


# ------------------------------------------------------ shared experts ----
def _shared_layer(seed=31, T=12, d=8, F=10, N=4, S=2):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, d))
    w_r = rng.normal(size=(N, d))
    W = {"w_gate": rng.normal(size=(N + S, F, d)) * 0.3, "w_up": rng.normal(size=(N + S, F, d)) * 0.3,
         "w_down": rng.normal(size=(N + S, d, F)) * 0.3}
    return x, w_r, W, (lambda e: O.stacked_expert(W, e))


def test_shared_experts_add_plain_ffns():
    """[替代FFN] §5 and §1: with shared experts the output gains, on every token,
    each shared expert's FFN(x) = W_down (silu(W_gate x) * (W_up x))."""
    x, w_r, W, ex = _shared_layer()
    base = O.moe_forward(x, w_r, None, ex, K=2, activation="swiglu")
    withs = O.moe_forward(x, w_r, None, ex, K=2, activation="swiglu", n_shared=2)
    direct = sum(((torch.nn.functional.silu(torch.from_numpy(x @ W["w_gate"][4 + s].T))).numpy()
                  * (x @ W["w_up"][4 + s].T)) @ W["w_down"][4 + s].T for s in range(2))
    assert np.max(np.abs(withs["y"] - base["y"] - direct)) < 1e-12
    # routing and statistics do not see the shared experts
    for k in ("idx", "gate", "count", "P", "kept", "offsets"):
        assert np.array_equal(base[k], withs[k])


def test_shared_experts_survive_zero_capacity():
    """Capacity drops only routed assignments: with C = 0 the output is the
    shared experts' sum (plus x with the residual)."""
    x, w_r, W, ex = _shared_layer(seed=32)
    r = O.moe_forward(x, w_r, None, ex, K=2, activation="swiglu", capacity_factor=0.01,
                      n_shared=2, add_residual=True)
    assert r["C"] == 0
    assert np.max(np.abs(r["y"] - x - O.shared_experts_output(x, ex, 4, 2, "swiglu"))) < 1e-12


def test_shared_expert_equals_always_routed_expert():
    """One shared expert is the same as an extra routed expert that every
    token picks with gate 1: a 2-expert layer whose router always picks
    expert 1 (K=1, renormalised gate = 1) over expert 0 equals a 1-expert
    layer whose expert 0 never fires (capacity 0) plus expert 1 as shared."""
    rng = np.random.default_rng(33)
    x = rng.normal(size=(9, 6))
    W = {"w_gate": rng.normal(size=(2, 7, 6)), "w_up": rng.normal(size=(2, 7, 6)),
         "w_down": rng.normal(size=(2, 6, 7))}
    ex = lambda e: O.stacked_expert(W, e)
    w_r = np.zeros((2, 6))
    b_r = np.array([0.0, 50.0])
    routed = O.moe_forward(x, w_r, b_r, ex, K=1, activation="swiglu")
    shared = O.moe_forward(x, np.zeros((1, 6)), None, ex, K=1, activation="swiglu",
                           capacity_factor=0.01, n_shared=1)
    assert np.max(np.abs(routed["y"] - shared["y"])) < 1e-12


def test_mutation_shared_gate_is_caught(monkeypatch):
    orig = O.shared_experts_output
    monkeypatch.setattr(O, "shared_experts_output",
                        lambda xs, ex, N, S, act: 0.5 * orig(xs, ex, N, S, act))
    with pytest.raises(AssertionError):
        test_shared_experts_add_plain_ffns()
