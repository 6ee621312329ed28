"""Expert-parallel exchange over two processes (gloo on the CPU, world size
2): "MoE 的核心思想", 前向传播中的 All-to-All 通信. Each rank routes and
dispatches its own half of one batch, packs its rows by destination, and the
ranks exchange them with all_to_all_single (split sizes from the all-gathered
per-expert counts); each rank regroups what it received by expert, runs the
experts it holds, regroups the outputs back, the second all_to_all_single
returns them, and each rank unpacks them into its slots and takes the
gate-weighted sum. Every rank's output must equal the single-device layer on
its own tokens. The arithmetic is the float64 oracle's; the exchange is a real
collective between processes."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, owner, wl_kwargs, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import moe_inputs
    from oracle import moe_oracle as O
    from oracle import moe_oracle_ep as E

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = moe_inputs.MoEWorkload("ep_gloo", **wl_kwargs)
        N, K = w.N, w.K
        x = moe_inputs.make_x(w, T=w.T * world)[rank * w.T:(rank + 1) * w.T]
        w_r, b_r = moe_inputs.make_router(w)
        experts = moe_inputs.make_experts(w, "cpu")
        expert_of = lambda e: {k: v[e] for k, v in experts.items()}
        # this rank's routing and capacity-limited dispatch
        l = O.router_logits(x, w_r, b_r)
        idx = O.topk_experts(l, K)
        gate = O.renormalised_gates(l, idx)
        disp = O.dispatch(idx, N, O.capacity(K, N, w.capacity_factor, w.T))
        x_perm = O.f64(x)[disp["token_of_slot"]]
        send, send_counts = E.pack(x_perm, disp["offsets"], owner, world)
        # every rank's per-expert counts, then the dispatch all-to-all
        kept = torch.from_numpy(disp["kept"].astype(np.int64))
        gathered = [torch.empty_like(kept) for _ in range(world)]
        dist.all_gather(gathered, kept)
        kept_all = torch.stack(gathered).numpy()
        mine = E.local_experts(owner, rank)
        recv_counts = [int(kept_all[s, mine].sum()) for s in range(world)]
        recv = torch.empty((sum(recv_counts), w.d), dtype=torch.float64)
        dist.all_to_all_single(recv, torch.from_numpy(np.ascontiguousarray(send)),
                               recv_counts, [int(c) for c in send_counts])
        # local compute on the experts this rank holds
        x_loc, loff = E.regroup(recv.numpy(), kept_all, owner, rank)
        o_loc = np.zeros_like(x_loc)
        for j, e in enumerate(mine):
            if loff[j + 1] > loff[j]:
                ew = {k: O.f64(v) for k, v in expert_of(int(e)).items()}
                o_loc[loff[j]:loff[j + 1]] = O.expert_apply(w.activation,
                                                            x_loc[loff[j]:loff[j + 1]], ew)
        back = E.regroup_back(o_loc, kept_all, owner, rank)
        # the combine all-to-all: outputs return in the order they were sent
        returned = torch.empty((int(send_counts.sum()), w.d), dtype=torch.float64)
        dist.all_to_all_single(returned, torch.from_numpy(np.ascontiguousarray(back)),
                               [int(c) for c in send_counts], recv_counts)
        o = E.unpack(returned.numpy(), disp["offsets"], owner, world)
        y = O.f64(x).copy() if w.add_residual else np.zeros((w.T, w.d))
        for t in range(w.T):
            for k in range(K):
                if disp["slot_of"][t, k] >= 0:
                    y[t] += gate[t, k] * o[disp["slot_of"][t, k]]
        ref = O.moe_forward(x, w_r, b_r, expert_of, K=K, activation=w.activation,
                            capacity_factor=w.capacity_factor, add_residual=w.add_residual)
        err = float(np.max(np.abs(y - ref["y"])))
        q.put((rank, err, float(np.abs(ref["y"]).max()), recv_counts,
               int(disp["n_dropped"])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("owner_name", ["block", "round_robin"])
def test_ep_exchange_over_two_gloo_ranks(owner_name):
    wl_kwargs = dict(T=96, d=16, F=24, N=6, K=2, init="uniform", capacity_factor=1.0,
                     add_residual=True, router_bias="skew")
    owner = (np.array([0, 0, 0, 1, 1, 1]) if owner_name == "block"
             else np.array([0, 1, 0, 1, 0, 1]))
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, owner, wl_kwargs, q))
             for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, *_ in results) == [0, 1]
    for rank, err, scale, recv_counts, dropped in results:
        assert err <= 1e-12 * max(1.0, scale), (rank, err)
        assert min(recv_counts) > 0        # both ranks really received rows from both
    assert sum(d for *_, d in results) > 0  # the capacity dropped something
