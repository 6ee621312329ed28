"""Expert-parallel staging on the GPU, through the C ABI ("MoE 的核心思想",
Expert Parallelism and 前向传播中的 All-to-All 通信).

Every layout the four calls write is compared bit for bit with the oracle's
(oracle/moe_oracle_ep.py). End to end, R source devices are emulated on one
GPU: each routes and dispatches its own part of a batch and packs it; the
test moves the packed blocks between the emulated devices (the all-to-all,
done here with tensor slices); each device regroups what it received, runs
its experts with moe_expert_ffn, regroups the outputs back; the blocks go
back; each source unpacks them and combines. Every source's y is checked
against the float64 oracle of the single-device layer on its tokens.
Device-detected errors (an owner out of range, a device receiving more rows
than its buffers hold) must leave the outputs untouched and set the status.
"""
import numpy as np
import pytest
import torch

import moe_inputs
from moe_inputs import MoEWorkload
from oracle import moe_oracle as O
from oracle import moe_oracle_ep as E

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mixture_experts_layer_101_b300 as moe
    import moe_testlib as L


def bits(t: torch.Tensor) -> np.ndarray:
    """The raw bit patterns of a tensor's rows (bf16 or fp32), for exact
    comparisons in numpy."""
    t = t.contiguous().cpu()
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)).numpy()


def source_device(cfg, inp):
    """Route and dispatch one source device's tokens; device tensors."""
    T, K, N, d = cfg.T, cfg.top_k, cfg.n_experts, cfg.d_model
    A = max(moe.a_max(cfg), 1)
    ws = moe.alloc_workspace(cfg)
    st = moe.Stats(N)
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    gate = torch.zeros((T, K), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, inp["x"], inp["w_r"], inp["b_r"], idx, gate, st, ws)
    offsets = torch.zeros(N + 1, dtype=torch.int32, device="cuda")
    slot_of = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    tos = torch.zeros(A, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((A, d), dtype=cfg.torch_dtype, device="cuda")
    moe.moe_dispatch(cfg, inp["x"], idx, offsets, slot_of, tos, x_perm, st, ws)
    return {"idx": idx, "gate": gate, "offsets": offsets, "slot_of": slot_of, "x_perm": x_perm,
            "stats": st, "A": A}


def split_inputs(w, R):
    """R source devices' inputs: consecutive parts of one batch of R*T tokens,
    the same router and experts."""
    x_all = moe_inputs.make_x(w, T=w.T * R)
    w_r, b_r = moe_inputs.make_router(w)
    experts = moe_inputs.make_experts(w, "cuda")
    return [{"x": x_all[r * w.T:(r + 1) * w.T].contiguous().cuda(), "w_r": w_r.cuda(),
             "b_r": None if b_r is None else b_r.cuda(), "experts": experts}
            for r in range(R)]


CASES = {
    "tc_block_4": (MoEWorkload("ep_tc", T=300, d=256, F=256, N=8, K=2), E.block_owner(8, 4), 4),
    "tc_round_robin_capacity": (MoEWorkload("ep_tc_cap", T=512, d=512, F=128, N=6, K=2,
                                            capacity_factor=1.0, add_residual=True,
                                            router_bias="skew"), np.arange(6) % 3, 3),
    "tc_rank_without_experts": (MoEWorkload("ep_tc_empty", T=200, d=256, F=128, N=4, K=1,
                                            add_residual=True), np.array([0, 0, 2, 2]), 3),
    "simt_gelu_fp32": (MoEWorkload("ep_simt", T=90, d=64, F=96, N=6, K=3, dtype="f32",
                                   activation="gelu", has_bias=True, init="uniform"),
                       np.array([1, 0, 1, 0, 1, 1]), 2),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_pack_and_unpack_match_the_oracle_bit_for_bit(name):
    w, owner, R = CASES[name]
    cfg = moe.LayerConfig.from_workload(w)
    inp = split_inputs(w, 1)[0]
    src = source_device(cfg, inp)
    own = torch.as_tensor(owner, dtype=torch.int32, device="cuda")
    ws = moe.alloc_ep_workspace(cfg, R)
    A, d = src["A"], w.d
    send = torch.zeros((A, d), dtype=cfg.torch_dtype, device="cuda")
    counts = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    st = moe.Stats(w.N)
    moe.moe_ep_pack(cfg, R, own, src["offsets"], src["x_perm"], send, counts, st, ws)
    torch.cuda.synchronize()
    assert st.status_bits() == 0
    offs = src["offsets"].cpu().numpy().astype(np.int64)
    n = int(offs[-1])
    ref_send, ref_counts = E.pack(bits(src["x_perm"])[:n], offs, owner, R)
    assert np.array_equal(counts.cpu().numpy(), ref_counts)
    assert np.array_equal(bits(send)[:n], ref_send)
    # unpack: arbitrary fp32 rows in send order back to their slots
    g = torch.Generator(device="cuda").manual_seed(3)
    back = torch.randn((A, d), generator=g, device="cuda")
    o = torch.zeros((A, d), dtype=torch.float32, device="cuda")
    moe.moe_ep_unpack(cfg, R, own, src["offsets"], back, o, st, ws)
    torch.cuda.synchronize()
    assert st.status_bits() == 0
    assert np.array_equal(bits(o)[:n], E.unpack(bits(back)[:n], offs, owner, R))


def exchange(blocks_by_source):
    """The all-to-all between the emulated devices: destination r receives
    every source's block for r, sources ascending."""
    R = len(blocks_by_source)
    return [torch.cat([blocks_by_source[s][r] for s in range(R)], dim=0) for r in range(R)]


def split(buf, counts):
    return list(torch.split(buf, [int(c) for c in counts], dim=0))


@pytest.mark.parametrize("name", sorted(CASES))
def test_ep_layer_over_emulated_devices(name):
    w, owner, R = CASES[name]
    N, K, d = w.N, w.K, w.d
    cfg = moe.LayerConfig.from_workload(w)
    inps = split_inputs(w, R)
    own = torch.as_tensor(owner, dtype=torch.int32, device="cuda")
    ws = moe.alloc_ep_workspace(cfg, R)
    st = moe.Stats(N)
    # dispatch step on every source: route, dispatch, pack
    srcs = []
    for inp in inps:
        src = source_device(cfg, inp)
        src["send"] = torch.zeros((src["A"], d), dtype=cfg.torch_dtype, device="cuda")
        src["counts"] = torch.zeros(R, dtype=torch.int32, device="cuda")
        moe.moe_ep_pack(cfg, R, own, src["offsets"], src["x_perm"], src["send"], src["counts"],
                        st, ws)
        src["counts_h"] = src["counts"].cpu().numpy()
        srcs.append(src)
    kept_all = torch.stack([s["stats"].kept for s in srcs]).contiguous()
    kept_h = kept_all.cpu().numpy().astype(np.int64)
    recv = exchange([split(s["send"][:int(s["counts_h"].sum())], s["counts_h"]) for s in srcs])
    # local compute on every destination
    back_blocks = []
    for r in range(R):
        mine = E.local_experts(owner, r)
        rows = int(recv[r].shape[0])
        cap = rows + 5                                   # buffers larger than needed
        recv_buf = torch.zeros((cap, d), dtype=cfg.torch_dtype, device="cuda")
        recv_buf[:rows] = recv[r]
        x_loc = torch.zeros((cap, d), dtype=cfg.torch_dtype, device="cuda")
        loff = torch.full((N + 1,), -1, dtype=torch.int32, device="cuda")
        moe.moe_ep_regroup(cfg, R, r, own, kept_all, cap, recv_buf, x_loc, loff, st, ws)
        torch.cuda.synchronize()
        ref_x, ref_loff = E.regroup(bits(recv_buf)[:rows], kept_h, owner, r)
        loff_h = loff.cpu().numpy()
        assert np.array_equal(loff_h[:len(mine) + 1], ref_loff)
        assert np.all(loff_h[len(mine):] == rows)
        assert np.array_equal(bits(x_loc)[:rows], ref_x)
        o_loc = torch.zeros((cap, d), dtype=torch.float32, device="cuda")
        if len(mine) > 0 and rows > 0:
            lcfg = moe.LayerConfig(T=cap, d_model=d, d_ff=w.F, n_experts=len(mine), top_k=1,
                                   dtype=w.dtype, activation=w.activation, has_bias=w.has_bias)
            sel = torch.as_tensor(mine, device="cuda")
            lw = {k: v.index_select(0, sel).contiguous() for k, v in inps[0]["experts"].items()}
            moe.moe_expert_ffn(lcfg, x_loc, loff[:len(mine) + 1].contiguous(), lw, o_loc, st,
                               moe.alloc_workspace(lcfg))
        back = torch.zeros((cap, d), dtype=torch.float32, device="cuda")
        moe.moe_ep_regroup_back(cfg, R, r, own, kept_all, cap, o_loc, back, st, ws)
        torch.cuda.synchronize()
        assert np.array_equal(bits(back)[:rows],
                              E.regroup_back(bits(o_loc)[:rows], kept_h, owner, r))
        from_each = [int(kept_h[s, mine].sum()) for s in range(R)]
        back_blocks.append(split(back[:rows], from_each))
    returned = exchange(back_blocks)
    # combine step on every source: unpack, gate-weighted sum
    for s, (src, inp) in enumerate(zip(srcs, inps)):
        A = src["A"]
        n = int(src["counts_h"].sum())
        back = torch.zeros((A, d), dtype=torch.float32, device="cuda")
        back[:n] = returned[s]
        o = torch.zeros((A, d), dtype=torch.float32, device="cuda")
        moe.moe_ep_unpack(cfg, R, own, src["offsets"], back, o, st, ws)
        y = torch.zeros((w.T, d), dtype=cfg.torch_dtype, device="cuda")
        moe.moe_combine(cfg, o, src["slot_of"], src["gate"], inp["x"], y)
        torch.cuda.synchronize()
        idx = src["idx"].cpu().numpy().astype(np.int64)
        x = inp["x"].cpu()
        b_r = None if inp["b_r"] is None else inp["b_r"].cpu()
        L.check_routing(O.router_logits(x, inp["w_r"].cpu(), b_r), idx, K)
        ref = O.moe_forward(x, inp["w_r"].cpu(), b_r, L.expert_reader(inp["experts"]), K=K,
                            activation=w.activation, capacity_factor=L.stored_cf(cfg),
                            add_residual=w.add_residual, idx_override=idx)
        assert np.array_equal(src["stats"].kept.cpu().numpy(), ref["kept"])
        rms = float(np.sqrt(np.mean(ref["y"] ** 2)))
        tol = L.y_tolerance(w.dtype) * rms
        assert float(np.max(np.abs(y.cpu().double().numpy() - ref["y"]))) <= tol
        if w.dtype == "bf16":
            assert L.stored_bar_excess(y.cpu(), ref["y"], tol) <= 0.0
    assert st.status_bits() == 0


def test_device_detected_errors_write_nothing():
    w, owner, R = CASES["tc_block_4"]
    cfg = moe.LayerConfig.from_workload(w)
    src = source_device(cfg, split_inputs(w, 1)[0])
    ws = moe.alloc_ep_workspace(cfg, R)
    A, d = src["A"], w.d
    # an owner outside [0, R): MOE_ERR_INDEX, send untouched
    bad_owner = torch.as_tensor(np.where(np.arange(w.N) == 5, R, owner), dtype=torch.int32,
                                device="cuda")
    send = torch.full((A, d), 7.0, dtype=cfg.torch_dtype, device="cuda")
    counts = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    st = moe.Stats(w.N)
    moe.moe_ep_pack(cfg, R, bad_owner, src["offsets"], src["x_perm"], send, counts, st, ws)
    torch.cuda.synchronize()
    assert st.status_bits() == 1 << moe.moe.MOE_ERR_INDEX
    assert (send == 7.0).all()
    # more rows than rows_cap: MOE_ERR_WORKSPACE, x_local untouched
    # (two sources with the same counts; device 0 holds the first half of the experts)
    own = torch.as_tensor(owner, dtype=torch.int32, device="cuda")
    kept_all = torch.stack([src["stats"].kept, src["stats"].kept]).contiguous()
    owner2 = E.block_owner(w.N, 2)
    need = int(kept_all.cpu().numpy()[:, E.local_experts(owner2, 0)].sum())
    cap = need - 1
    x_loc = torch.full((cap, d), 7.0, dtype=cfg.torch_dtype, device="cuda")
    recv = torch.zeros((cap, d), dtype=cfg.torch_dtype, device="cuda")
    loff = torch.zeros(w.N + 1, dtype=torch.int32, device="cuda")
    st2 = moe.Stats(w.N)
    ws2 = moe.alloc_ep_workspace(cfg, 2)
    own2 = torch.as_tensor(owner2, dtype=torch.int32, device="cuda")
    moe.moe_ep_regroup(cfg, 2, 0, own2, kept_all, cap, recv, x_loc, loff, st2, ws2)
    torch.cuda.synchronize()
    assert st2.status_bits() == 1 << moe.moe.MOE_ERR_WORKSPACE
    assert (x_loc == 7.0).all()
    # host-side errors: nothing launched
    with pytest.raises(moe.MoEError) as e:
        moe.moe_ep_pack(cfg, 0, own, src["offsets"], src["x_perm"], send, counts, st, ws)
    assert e.value.code == moe.moe.MOE_ERR_INVALID
    with pytest.raises(moe.MoEError) as e:
        moe.moe_ep_regroup(cfg, R, R, own, kept_all, 10, recv, x_loc, loff, st, ws)
    assert e.value.code == moe.moe.MOE_ERR_INVALID
