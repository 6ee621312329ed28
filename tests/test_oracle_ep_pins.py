"""Pins of the expert-parallel staging oracle (oracle/moe_oracle_ep.py).

"MoE 的核心思想", Expert Parallelism and 前向传播中的 All-to-All 通信: the
experts are spread over devices; tokens go to the device holding their expert
(dispatch all-to-all), each device runs its own experts (local compute), and
the outputs return to the source devices where the gate-weighted sum is taken
(combine all-to-all). Whatever the layout, the layer's output must be the
single-device layer's: the end-to-end pin runs R source devices' batches
through pack -> all-to-all -> regroup -> local experts -> regroup back ->
all-to-all -> unpack -> combine and compares each device's y with the
single-device oracle on its own tokens. The layout functions are also pinned
by brute force (stable sorts on the layout's keys) and by their inverses;
planted mistakes must be caught.
"""
import numpy as np
import pytest

import moe_inputs
from moe_inputs import MoEWorkload
from oracle import moe_oracle as O
from oracle import moe_oracle_ep as E


def random_offsets(rng, N, max_rows=9):
    kept = rng.integers(0, max_rows, size=N)
    return np.concatenate([[0], np.cumsum(kept)]).astype(np.int64)


OWNERS = {
    "block_4_of_8": (E.block_owner(8, 4), 4),
    "round_robin_3_of_7": (np.arange(7) % 3, 3),
    "rank_without_experts": (np.array([0, 0, 2, 2, 0, 2]), 3),
    "one_rank": (np.zeros(5, dtype=np.int64), 1),
    "one_expert_per_rank": (np.arange(6), 6),
}


def test_block_owner():
    assert list(E.block_owner(8, 4)) == [0, 0, 1, 1, 2, 2, 3, 3]
    assert list(E.block_owner(8, 8)) == list(range(8))
    assert list(E.block_owner(5, 1)) == [0] * 5
    assert list(E.block_owner(7, 3)) == [0, 0, 0, 1, 1, 2, 2]
    o = E.block_owner(256, 8)
    assert all(int((o == r).sum()) == 32 for r in range(8))
    assert np.all(np.diff(o) >= 0)


@pytest.mark.parametrize("name", sorted(OWNERS))
def test_pack_is_a_stable_sort_by_destination(name):
    owner, R = OWNERS[name]
    rng = np.random.default_rng(1)
    offsets = random_offsets(rng, len(owner))
    rows = rng.normal(size=(int(offsets[-1]), 3))
    send, counts = E.pack(rows, offsets, owner, R)
    # brute force: each slot's (destination, expert) key, stably sorted
    e_of_slot = np.searchsorted(offsets, np.arange(offsets[-1]), side="right") - 1
    order = np.lexsort((e_of_slot, owner[e_of_slot]))
    assert np.array_equal(send, rows[order])
    assert np.array_equal(counts, np.bincount(owner[e_of_slot], minlength=R))
    assert counts.sum() == offsets[-1]
    # unpack inverts pack
    assert np.array_equal(E.unpack(send, offsets, owner, R), rows)


def test_one_rank_pack_is_the_identity():
    owner, R = OWNERS["one_rank"]
    rng = np.random.default_rng(2)
    offsets = random_offsets(rng, len(owner))
    rows = rng.normal(size=(int(offsets[-1]), 4))
    send, counts = E.pack(rows, offsets, owner, R)
    assert np.array_equal(send, rows) and list(counts) == [offsets[-1]]


@pytest.mark.parametrize("name", sorted(OWNERS))
def test_regroup_is_a_stable_sort_by_expert_and_inverts(name):
    owner, R = OWNERS[name]
    N = len(owner)
    rng = np.random.default_rng(3)
    kept_all = rng.integers(0, 6, size=(R, N))
    for r in range(R):
        mine = E.local_experts(owner, r)
        # receive buffer: rows labelled (source, expert, i), source-major
        labels = [(s, int(e), i) for s in range(R) for e in mine for i in range(kept_all[s, e])]
        recv = np.array([[s, e, i] for (s, e, i) in labels], dtype=np.float64).reshape(-1, 3)
        x_local, loff = E.regroup(recv, kept_all, owner, r)
        order = sorted(range(len(labels)), key=lambda j: (labels[j][1], labels[j][0]))
        assert np.array_equal(x_local, recv[order])
        assert np.array_equal(np.diff(loff), kept_all[:, mine].sum(axis=0))
        assert np.array_equal(E.regroup_back(x_local, kept_all, owner, r), recv)


def _expert_of(experts):
    return lambda e: {k: v[e] for k, v in experts.items()}


def ep_layer(xs_by_rank, w_r, b_r, expert_of, owner, *, K, activation, cf, residual):
    """The layer over R devices through the EP staging, every step in the
    oracle: returns each source device's y."""
    R, N = len(xs_by_rank), w_r.shape[0]
    src = []
    for x in xs_by_rank:
        l = O.router_logits(x, w_r, b_r)
        idx = O.topk_experts(l, K)
        gate = O.renormalised_gates(l, idx)
        disp = O.dispatch(idx, N, O.capacity(K, N, cf, x.shape[0]))
        x_perm = O.f64(x)[disp["token_of_slot"]]
        send, counts = E.pack(x_perm, disp["offsets"], owner, R)
        src.append({"x": O.f64(x), "gate": gate, "disp": disp, "send": send,
                    "counts": counts})
    kept_all = np.stack([s["disp"]["kept"] for s in src])
    recv = E.exchange([E.split_by_counts(s["send"], s["counts"]) for s in src])
    back_blocks = []
    for r in range(R):
        x_loc, loff = E.regroup(recv[r], kept_all, owner, r)
        o_loc = np.zeros_like(x_loc)
        for j, e in enumerate(E.local_experts(owner, r)):
            if loff[j + 1] > loff[j]:
                ew = {k: O.f64(v) for k, v in expert_of(int(e)).items()}
                o_loc[loff[j]:loff[j + 1]] = O.expert_apply(activation, x_loc[loff[j]:loff[j + 1]],
                                                            ew)
        back = E.regroup_back(o_loc, kept_all, owner, r)
        from_each = [int(kept_all[s, E.local_experts(owner, r)].sum()) for s in range(R)]
        back_blocks.append(E.split_by_counts(back, from_each))
    returned = E.exchange(back_blocks)
    ys = []
    for s, d in enumerate(src):
        o = E.unpack(returned[s], d["disp"]["offsets"], owner, R)
        slot_of = d["disp"]["slot_of"]
        y = d["x"].copy() if residual else np.zeros_like(d["x"])
        for t in range(y.shape[0]):
            for k in range(K):
                if slot_of[t, k] >= 0:
                    y[t] += d["gate"][t, k] * o[slot_of[t, k]]
        ys.append(y)
    return ys


CASES = [
    # (workload, owner, R)
    (MoEWorkload("ep_block", T=96, d=16, F=24, N=8, K=2, init="uniform"),
     E.block_owner(8, 4), 4),
    (MoEWorkload("ep_round_robin_capacity", T=120, d=16, F=24, N=6, K=2, init="uniform",
                 capacity_factor=1.0, add_residual=True, router_bias="skew"),
     np.arange(6) % 4, 4),
    (MoEWorkload("ep_empty_rank_gelu", T=80, d=8, F=12, N=5, K=3, init="uniform",
                 activation="gelu", has_bias=True),
     np.array([0, 2, 2, 0, 2]), 3),
    (MoEWorkload("ep_top1", T=64, d=8, F=16, N=4, K=1, init="uniform", capacity_factor=1.25,
                 add_residual=True), E.block_owner(4, 2), 2),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_ep_layer_equals_single_device_layer(case):
    w, owner, R = case
    # one global batch split over the R devices (data-parallel sources)
    x_all = moe_inputs.make_x(w, T=w.T * R)
    xs = [x_all[r * w.T:(r + 1) * w.T] for r in range(R)]
    w_r, b_r = moe_inputs.make_router(w)
    experts = moe_inputs.make_experts(w, "cpu")
    ys = ep_layer(xs, w_r, b_r, _expert_of(experts), owner, K=w.K, activation=w.activation,
                  cf=w.capacity_factor, residual=w.add_residual)
    for r in range(R):
        ref = O.moe_forward(xs[r], w_r, b_r, _expert_of(experts), K=w.K,
                            activation=w.activation, capacity_factor=w.capacity_factor,
                            add_residual=w.add_residual)
        scale = max(1.0, float(np.abs(ref["y"]).max()))
        assert np.allclose(ys[r], ref["y"], rtol=0, atol=1e-12 * scale)


# ------------------------------------------- mutations caught by pins ----
def test_mutation_regroup_left_source_major_is_caught(monkeypatch):
    def wrong(recv, kept_all, owner, r):  # experts' rows not gathered across sources
        _, loff = orig(recv, kept_all, owner, r)
        return np.asarray(recv), loff
    orig = E.regroup
    monkeypatch.setattr(E, "regroup", wrong)
    with pytest.raises(AssertionError):
        test_ep_layer_equals_single_device_layer(CASES[0])


def test_mutation_destinations_reversed_in_pack_is_caught(monkeypatch):
    def wrong(rows, offsets, owner, R):
        blocks = [np.asarray(rows)[offsets[e]:offsets[e + 1]]
                  for r in reversed(range(R)) for e in E.local_experts(owner, r)]
        return np.concatenate(blocks, axis=0), E.send_counts(np.diff(offsets), owner, R)
    monkeypatch.setattr(E, "pack", wrong)
    with pytest.raises(AssertionError):
        test_pack_is_a_stable_sort_by_destination("block_4_of_8")


def test_mutation_unpack_in_slot_order_is_caught(monkeypatch):
    # returned rows taken as if they were already in slot order: right only
    # when the placement keeps experts in ascending order across ranks
    monkeypatch.setattr(E, "unpack", lambda back, offsets, owner, R, n_rows=None:
                        np.asarray(back))
    with pytest.raises(AssertionError):
        test_ep_layer_equals_single_device_layer(CASES[1])
