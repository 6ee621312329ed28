"""The layer at the largest supported batch, T = 2^24 tokens (K = 2 of N = 8,
no capacity limit, so 2^25 assignments): every index the kernels form stays
in range there.

Every token: the expert counts, the offsets, the slot of every assignment and
the token of every slot are checked against their defining properties (the
rank-major visiting order of the dispatch); the selection statistic P against
float64 logits computed in chunks. A sample of tokens: top-K indices, gates
and y against the float64 oracle run on those tokens.
"""
import numpy as np
import pytest
import torch

import moe_inputs
from moe_inputs import MoEWorkload
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mixture_experts_layer_101_b300 as moe
    import moe_testlib as L

T_MAX = 1 << 24


def test_max_tokens_layer():
    w = MoEWorkload("max_tokens", T=T_MAX, d=64, F=32, N=8, K=2)
    T, d, N, K = w.T, w.d, w.N, w.K
    cfg = moe.LayerConfig.from_workload(w)
    x = moe_inputs.make_x(w, device="cuda")
    w_r, b_r = moe_inputs.make_router(w)
    experts = moe_inputs.make_experts(w, "cuda")
    ws = moe.alloc_workspace(cfg)
    st = moe.Stats(N)
    idx = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    gate = torch.zeros((T, K), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, x, w_r.cuda(), None, idx, gate, st, ws)
    A = T * K
    offsets = torch.zeros(N + 1, dtype=torch.int32, device="cuda")
    slot_of = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    tos = torch.full((A,), -7, dtype=torch.int32, device="cuda")
    x_perm = torch.empty((A, d), dtype=x.dtype, device="cuda")
    moe.moe_dispatch(cfg, x, idx, offsets, slot_of, tos, x_perm, st, ws)
    o = torch.empty((A, d), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(cfg, x_perm, offsets, experts, o, st, ws)
    y = torch.empty((T, d), dtype=x.dtype, device="cuda")
    moe.moe_combine(cfg, o, slot_of, gate, x, y)
    torch.cuda.synchronize()
    stats = st.to_host()
    assert stats["status"] == 0
    del x_perm, o, ws
    idx_h = idx.cpu().numpy().astype(np.int64)
    slot_h = slot_of.cpu().numpy().astype(np.int64)
    tos_h = tos.cpu().numpy().astype(np.int64)
    off_h = offsets.cpu().numpy().astype(np.int64)

    # counts, offsets (no capacity: everything kept, nothing dropped)
    assert idx_h.min() >= 0 and idx_h.max() < N
    assert np.all(idx_h[:, 0] != idx_h[:, 1])
    count = np.bincount(idx_h.ravel(), minlength=N)
    assert np.array_equal(stats["count"], count)
    assert np.array_equal(stats["kept"], count) and stats["n_dropped"] == 0
    assert np.array_equal(off_h, np.concatenate([[0], np.cumsum(count)]))
    # dispatch order: slots of expert e list its assignments (k, t) in rank-major order
    q = np.arange(K * T, dtype=np.int64)              # visiting order q = k*T + t
    e_of_q = idx_h.T.ravel()                          # expert of assignment q
    order = np.argsort(e_of_q, kind="stable")         # by expert, q ascending within
    assert np.array_equal(tos_h, order % T)
    want_slot = np.empty(K * T, dtype=np.int64)
    want_slot[order] = np.arange(K * T)
    assert np.array_equal(slot_h, want_slot.reshape(K, T).T)
    del q, e_of_q, order, want_slot

    # P against float64 logits over every token, in chunks of 2^20 tokens
    psum = np.zeros(N)
    for c0 in range(0, T, 1 << 20):
        l64 = O.router_logits(x[c0:c0 + (1 << 20)].cpu(), w_r, None)
        psum += O.softmax(l64).sum(axis=0)
    assert np.allclose(stats["P"], psum / T, rtol=L.STAT_RTOL, atol=1e-7)

    # sampled tokens (first, last, random): routing, gates and y against the
    # oracle. Without a capacity limit a token's output depends on that token
    # alone, so the oracle runs the sampled tokens as a batch of their own
    # (on the GPU's routing, which check_routing accepted first).
    rng = np.random.default_rng(7)
    tok = np.unique(np.concatenate([[0, 1, T - 2, T - 1], rng.choice(T, 60, replace=False)]))
    tt = torch.from_numpy(tok).cuda()
    xs = x[tt].cpu()
    L.check_routing(O.router_logits(xs, w_r, None), idx_h[tok], K)
    ref = O.moe_forward(xs, w_r, None, L.expert_reader(experts), K=K,
                        activation=w.activation, idx_override=idx_h[tok])
    assert np.max(np.abs(gate[tt].cpu().numpy() - ref["gate"])) <= L.GATE_TOL
    y_tok = y[tt].cpu()
    rms = float(np.sqrt(np.mean(ref["y"] ** 2)))
    tol = L.y_tolerance(cfg.dtype) * rms
    assert np.max(np.abs(y_tok.double().numpy() - ref["y"])) <= tol
    assert L.stored_bar_excess(y_tok, ref["y"], tol) <= 0.0
