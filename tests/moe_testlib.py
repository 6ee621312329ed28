"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI (stage by stage, or whole), and compare with the float64 oracle.

Comparison rules:
  * routing: bit-exact expert indices except on near-tie tokens (some adjacent
    gap among the K+1 largest float64 logits below 1e-5); a near-tie token's
    GPU choice is accepted when each chosen expert's float64 logit lies within
    1e-5 of the oracle's choice at the same rank; everything downstream is then
    compared against the oracle re-run on the GPU's routing;
  * counts, kept, offsets, slots, token order and the drop set: bit-exact;
  * gates: |err| <= 1e-5; P and L_aux: relative error <= 1e-5;
  * y, fp32 layers: max |err| <= 1e-4 * rms(y);
  * y, bf16 layers, three checks:
      - the stated bar on the value y is rounded from: every y_gpu element is
        the bf16 rounding of some value within 2e-2 * rms(y) of the exact y,
        i.e. y lies within 2e-2 * rms(y) of the interval of reals that round
        to y_gpu (stored_bar_excess); the bf16 storage of y alone can be off
        by 2^-8 |y|, which at the largest |y| of a 16-million-element output
        (about 5.5 rms) is already 0.021 rms;
      - the per-element bound of the bf16 roundings the path performs
        (bf16_rounding_bound: h and y rounded once each);
      - the raw bar max |err| <= 2e-2 * rms(y) (strict=True), for the layers
        whose outputs meet it; the others are listed with their measured
        ratios where they are tested.
"""
from __future__ import annotations

import numpy as np
import torch

import mixture_experts_layer_101_b300 as moe
import moe_inputs
from oracle import moe_oracle as O
from oracle import moe_oracle_grad as OG

NEAR_TIE_EPS = 1e-5
BF16_U = 2.0 ** -8   # unit roundoff of bf16 round-to-nearest (8 significant bits)
GATE_TOL = 1e-5
STAT_RTOL = 1e-5


def stored_cf(cfg) -> float:
    """The capacity factor as the layer stores it (moe_config carries a
    float32), which is the value the oracle must be given: e.g. 0.9f is just
    below 0.9, so floor(2 * 0.9f * 3000 / 4) = 1349 where the double 0.9 gives
    1350."""
    return float(np.float32(cfg.capacity_factor))


def y_tolerance(dtype: str) -> float:
    return 1e-4 if dtype == "f32" else 2e-2


def bf16_neighbours(v: torch.Tensor):
    """The bf16 values just below and just above each element of the bf16
    tensor v (as float64 numpy arrays), by stepping its bit pattern; zero's
    neighbours are the smallest subnormals."""
    bits = v.contiguous().view(torch.int16).to(torch.int32)
    neg = bits < 0
    mag = bits & 0x7FFF
    up_mag = torch.where(neg, mag - 1, mag + 1)      # towards +inf
    dn_mag = torch.where(neg, mag + 1, mag - 1)      # towards -inf
    # zero (either sign): the neighbours are +-smallest subnormal
    zero = mag == 0
    up_bits = torch.where(zero, torch.ones_like(bits), torch.where(neg, up_mag | 0x8000, up_mag))
    dn_bits = torch.where(zero, torch.full_like(bits, 0x8001),
                          torch.where(neg, dn_mag | 0x8000, dn_mag))
    as_bf16 = lambda b: (b & 0xFFFF).to(torch.int16).view(torch.bfloat16).double().numpy()
    return as_bf16(dn_bits), as_bf16(up_bits)


def stored_bar_excess(y_gpu: torch.Tensor, y_ref: np.ndarray, tol: float) -> float:
    """max over elements of the distance (beyond tol) from the exact y to the
    interval of reals that round to y_gpu in bf16 (round to nearest: half the
    gap to each neighbour). <= 0 means every y_gpu element is the rounding of
    some value within tol of y."""
    v = y_gpu.double().numpy()
    dn, up = bf16_neighbours(y_gpu)
    lo = v - (v - dn) / 2.0
    hi = v + (up - v) / 2.0
    dist = np.maximum(lo - y_ref, y_ref - hi)
    return float(np.max(dist - tol, initial=-np.inf))


def device_inputs(w: moe_inputs.MoEWorkload):
    """Inputs on cuda:0; x and the router drawn on the CPU, experts on the GPU."""
    x = moe_inputs.make_x(w)
    w_r, b_r = moe_inputs.make_router(w)
    sb = moe_inputs.make_select_bias(w)
    experts = moe_inputs.make_experts(w, "cuda")
    return {"x": x.cuda(), "w_r": w_r.cuda(), "b_r": None if b_r is None else b_r.cuda(),
            "select_bias": None if sb is None else sb.cuda(), "experts": experts}


def layer_config(w: moe_inputs.MoEWorkload, inp: dict) -> moe.LayerConfig:
    cfg = moe.LayerConfig.from_workload(w)
    cfg.select_bias = inp.get("select_bias")
    return cfg


def expert_reader(experts: dict):
    """expert_of(e) for the oracle: copies expert e's weights to the host."""
    return lambda e: {k: v[e].cpu() for k, v in experts.items()}


def run_stages(cfg: moe.LayerConfig, inp: dict, ws_fill: int | None = None) -> dict:
    """route -> dispatch -> expert_ffn -> combine through the C ABI (with
    ws_fill, every workspace byte is set to it first)."""
    dev = "cuda"
    T, K, N, d = cfg.T, cfg.top_k, cfg.n_experts, cfg.d_model
    S = cfg.n_shared
    A = moe.rows_max(cfg)
    ws = moe.alloc_workspace(cfg)
    if ws_fill is not None:
        ws.fill_(ws_fill)
    st = moe.Stats(N)
    idx = torch.full((T, K), -7, dtype=torch.int32, device=dev)
    gate = torch.zeros((T, K), dtype=torch.float32, device=dev)
    moe.moe_route(cfg, inp["x"], inp["w_r"], inp["b_r"], idx, gate, st, ws)
    offsets = torch.zeros(N + S + 1, dtype=torch.int32, device=dev)
    slot_of = torch.full((T, K + S), -7, dtype=torch.int32, device=dev)
    tos = torch.full((max(A, 1),), -7, dtype=torch.int32, device=dev)
    x_perm = torch.zeros((max(A, 1), d), dtype=cfg.torch_dtype, device=dev)
    moe.moe_dispatch(cfg, inp["x"], idx, offsets, slot_of, tos, x_perm, st, ws)
    o = torch.zeros((max(A, 1), d), dtype=torch.float32, device=dev)
    moe.moe_expert_ffn(cfg, x_perm, offsets, inp["experts"], o, st, ws)
    y = torch.zeros((T, d), dtype=cfg.torch_dtype, device=dev)
    moe.moe_combine(cfg, o, slot_of, gate, inp["x"], y)
    torch.cuda.synchronize()
    out = {"idx": idx, "gate": gate, "offsets": offsets, "slot_of": slot_of,
           "token_of_slot": tos, "x_perm": x_perm, "o": o, "y": y}
    out = {k: v.cpu() for k, v in out.items()}
    out["stats"] = st.to_host()
    return out


def run_forward(cfg: moe.LayerConfig, inp: dict):
    layer = moe.MoELayer(cfg, inp["w_r"], inp["b_r"], inp["experts"])
    y = layer.forward(inp["x"]).clone()
    torch.cuda.synchronize()
    return y.cpu(), layer.stats.to_host()


def check_routing(l64: np.ndarray, idx_gpu: np.ndarray, K: int):
    """Returns (near-tie token count, tokens whose routing differs)."""
    idx_o = O.topk_experts(l64, K)
    near = O.near_tie_tokens(l64, K, NEAR_TIE_EPS)
    diff = np.any(idx_gpu != idx_o, axis=1)
    bad = diff & ~near
    assert not bad.any(), f"routing differs on {bad.sum()} tokens without a near-tie"
    for t in np.nonzero(diff)[0]:
        assert len(set(idx_gpu[t].tolist())) == K
        assert np.all(np.abs(l64[t, idx_gpu[t]] - l64[t, idx_o[t]]) < NEAR_TIE_EPS)
    return int(near.sum()), int(diff.sum())


def bf16_rounding_bound(cfg: moe.LayerConfig, inp: dict, ref: dict) -> np.ndarray:
    """Per-element bound [len(tokens)][d] on |y_gpu - y| that bf16 storage
    alone allows, with the unit roundoff of bf16 round-to-nearest u = 2^-8
    (8 significant bits): h is rounded to bf16 once (relative error <= u per
    element, which reaches o as at most u * sum_f |W_down[j, f]| |h_f|), y is
    rounded to bf16 once (<= u |y|), plus 1e-3 * rms(y) for fp32 accumulation
    order and gate rounding."""
    x = O.f64(inp["x"])
    tok = ref["tokens"]
    bound = np.zeros((len(tok), cfg.d_model))
    reader = expert_reader(inp["experts"])
    rows = {}
    for i, t in enumerate(tok):
        for k in range(cfg.top_k):
            if ref["slot_of"][t, k] >= 0:
                rows.setdefault(int(ref["idx"][t, k]), []).append((i, int(t), k))
    for s in range(cfg.n_shared):  # shared experts: every token, gate 1
        for i, t in enumerate(tok):
            rows.setdefault(cfg.n_experts + s, []).append((i, int(t), -1))
    for e, lst in rows.items():
        ew = {kk: O.f64(v) for kk, v in reader(e).items() if v is not None}
        xe = x[[t for (_, t, _) in lst]]
        if cfg.activation == "swiglu":
            h = O.silu(xe @ ew["w_gate"].T) * (xe @ ew["w_up"].T)
            wd = ew["w_down"]
        else:
            z = xe @ ew["w1"].T + (ew["b1"][None, :] if "b1" in ew else 0.0)
            h = O.gelu_erf(z)
            wd = ew["w2"]
        scale = np.abs(h) @ np.abs(wd).T * BF16_U
        for r, (i, t, k) in enumerate(lst):
            bound[i] += (ref["gate"][t, k] if k >= 0 else 1.0) * scale[r]
    y = ref["y"]
    rms = float(np.sqrt(np.mean(y ** 2))) if y.size else 0.0
    return bound + 2.0 ** -8 * np.abs(y) + 1e-3 * rms


def check_layer(cfg: moe.LayerConfig, inp: dict, gpu: dict, *, tokens=None,
                strict: bool = True, stored: bool = True):
    """Compare a stage-wise GPU run against the oracle. tokens: the tokens
    whose y is checked (None = all); routing, statistics and dispatch always
    cover every token. bf16 layers always meet the per-element rounding
    bound; strict: also max |err| <= 2e-2 * rms(y) on the raw output; stored:
    also the 2e-2 * rms(y) bar on the value y is rounded from (see the module
    notes). Returns a summary dict (near-tie tokens, tokens whose routing
    differs from the oracle's, max |err| / rms(y), ...)."""
    K, N = cfg.top_k, cfg.n_experts
    x, w_r, b_r = inp["x"].cpu(), inp["w_r"].cpu(), None if inp["b_r"] is None else inp["b_r"].cpu()
    sb = None if cfg.select_bias is None else cfg.select_bias.cpu()
    l64 = O.router_logits(x, w_r, b_r)
    key64 = l64 if sb is None else l64 + O.f64(sb)[None, :]  # what the top-K compares
    idx_gpu = gpu["idx"].numpy().astype(np.int64)
    n_near, n_diff = check_routing(key64, idx_gpu, K)
    ref = O.moe_forward(x, w_r, b_r, expert_reader(inp["experts"]), K=K,
                        activation=cfg.activation, capacity_factor=stored_cf(cfg),
                        alpha=cfg.alpha, add_residual=cfg.add_residual, tokens=tokens,
                        idx_override=idx_gpu, gate_mode=cfg.gate_mode, select_bias=sb,
                        n_shared=cfg.n_shared)
    # gates and statistics
    assert np.max(np.abs(gpu["gate"].numpy() - ref["gate"]), initial=0) <= GATE_TOL
    st = gpu["stats"]
    assert np.array_equal(st["count"], ref["count"])
    assert np.allclose(st["P"], ref["P"], rtol=STAT_RTOL, atol=1e-7)
    assert np.allclose(st["f"], ref["f"], rtol=1e-6, atol=0)
    assert abs(st["l_aux"] - ref["l_aux"]) <= STAT_RTOL * abs(ref["l_aux"]) + 1e-9
    assert abs(st["z_loss"] - ref["z_loss"]) <= STAT_RTOL * abs(ref["z_loss"]) + 1e-6
    assert abs(st["entropy"] - ref["entropy"]) <= STAT_RTOL * abs(ref["entropy"]) + 1e-6
    assert st["status"] == 0
    # dispatch: bit-exact
    assert np.array_equal(st["kept"], ref["kept"]), (st["kept"], ref["kept"])
    assert st["n_dropped"] == ref["n_dropped"]
    S, T = cfg.n_shared, cfg.T
    offs = gpu["offsets"].numpy()
    assert np.array_equal(offs[:N + 1], ref["offsets"])
    A = int(ref["offsets"][-1])
    assert np.array_equal(offs[N:], A + T * np.arange(S + 1))   # shared experts: T rows each
    assert np.array_equal(gpu["slot_of"].numpy()[:, :K], ref["slot_of"])
    for s in range(S):
        assert np.array_equal(gpu["slot_of"].numpy()[:, K + s], A + s * T + np.arange(T))
    assert np.array_equal(gpu["token_of_slot"].numpy()[:A], ref["token_of_slot"])
    if A > 0:
        tos = torch.from_numpy(ref["token_of_slot"])
        assert torch.equal(gpu["x_perm"][:A], inp["x"].cpu()[tos])
    for s in range(S):
        assert torch.equal(gpu["x_perm"][A + s * T:A + (s + 1) * T], inp["x"].cpu())
    # outputs
    tok = ref["tokens"]
    y_gpu = gpu["y"].double().numpy()[tok]
    y_ref = ref["y"]
    rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    err = float(np.max(np.abs(y_gpu - y_ref))) if y_ref.size else 0.0
    tol = y_tolerance(cfg.dtype) * rms
    if cfg.dtype == "bf16":
        # the stated bar on the value the stored y was rounded from
        if stored:
            excess_stored = stored_bar_excess(gpu["y"][torch.as_tensor(tok)], y_ref, tol)
            assert excess_stored <= 0.0, ("stored bar", err, rms, excess_stored)
        # per-element bound from the bf16 roundings the path performs
        excess = np.abs(y_gpu - y_ref) - bf16_rounding_bound(cfg, inp, ref)
        assert excess.max(initial=-1.0) <= 0.0, ("rounding bound", err, rms,
                                                 float(excess.max()))
    if cfg.dtype != "bf16" or strict:
        assert err <= tol + 1e-30, ("raw bar", err, rms, err / rms if rms > 0 else 0.0)
    return {"near_ties": n_near, "routing_diff": n_diff, "A": A, "y_err_over_rms":
            err / rms if rms > 0 else 0.0, "n_dropped": ref["n_dropped"]}


# --------------------------------------------------------------- backward ----
GRAD_TOL_F32 = 1e-4   # fp32 layers: max |err| <= 1e-4 * rms, as for y


def _silu_parts(a):
    s = 1.0 / (1.0 + np.exp(-a))
    silu = a * s
    d1 = s * (1.0 + a * (1.0 - s))
    d2 = s * (1.0 - s) * (2.0 + a * (1.0 - 2.0 * s))
    return silu, d1, d2


def grad_rounding_bounds(cfg: moe.LayerConfig, inp: dict, dy, ref: dict) -> dict:
    """First-order per-element bounds on |gradient_gpu - gradient| that the
    bf16 roundings of a bf16 SwiGLU layer allow (u = 2^-8 per rounding):
      do = g dy rounded (u |do|); the forward's h rounded (u |h|); the kept
      pre-activations a, b rounded (u |a|, u |b|); the pre-activation
      gradients da = dh b silu'(a), db = dh silu(a) rounded (u |da|, u |db|).
    Propagated: E_dh = E_do |W_down|; E_da = u|da| + |b silu'(a)| E_dh +
    |dh b silu''(a)| E_a + |dh silu'(a)| E_b; E_db = u|db| + |silu(a)| E_dh +
    |dh silu'(a)| E_a; E_dW_down = E_do^T |h| + |do|^T E_h; E_dW_gate =
    E_da^T |x|; E_dW_up = E_db^T |x|; E_dx_perm = E_da |W_gate| + E_db |W_up|;
    through the gate gradient dg = <dy, o> with E_o = E_h |W_down|^T into the
    logit gradient (renormalised gates: E_dl[i_k] = g_k (E_dg_k + sum g E_dg);
    full-softmax gates: E_dl = p (E_dp + <p, E_dp>)), then E_dx += E_dl
    |W_r| and E_dW_r = E_dl^T |x|. Each bound gets 1e-3 * rms of its
    reference added for fp32 accumulation order and transcendental rounding.
    Returns {"dx": [len(tokens)][d], "dw_r": [N][d], "db_r": [N],
    "dw_gate": {e: [F][d]}, ...} for the tokens / experts in ref."""
    u = BF16_U
    K, N, S = cfg.top_k, cfg.n_experts, cfg.n_shared
    fwd = ref["fwd"]
    xs = O.f64(inp["x"])
    dys = O.f64(dy)
    T = xs.shape[0]
    gate, idx, slot_of, p = fwd["gate"], fwd["idx"], fwd["slot_of"], fwd["p"]
    reader = expert_reader(inp["experts"])
    tok = ref["tokens"]
    tok_pos = {int(t): i for i, t in enumerate(tok)}
    E_dxp_tok = np.zeros((len(tok), xs.shape[1]))
    E_dg = np.zeros((T, K))
    bounds = {"dw_gate": {}, "dw_up": {}, "dw_down": {}}
    # rows to evaluate: every row of an expert whose weight gradient is
    # compared, and the rows of the compared tokens (all tokens when the
    # router gradients are compared, which need every gate gradient)
    all_rows = "dw_r" in ref
    wanted = set(ref["dw"])
    rows_of = {}
    for t in range(T):
        for k in range(K):
            if slot_of[t, k] >= 0:
                e = int(idx[t, k])
                if all_rows or e in wanted or t in tok_pos:
                    rows_of.setdefault(e, []).append((t, k))
    for s_ in range(S):
        ts = range(T) if (all_rows or N + s_ in wanted) else [int(t) for t in tok]
        rows_of[N + s_] = [(t, -1) for t in ts]
    for e, rows in rows_of.items():
        ew = {kk: O.f64(v) for kk, v in reader(e).items() if v is not None}
        ts = [t for t, _ in rows]
        g = np.array([gate[t, k] if k >= 0 else 1.0 for t, k in rows])
        xe = xs[ts]
        a, b = xe @ ew["w_gate"].T, xe @ ew["w_up"].T
        silu, d1, d2 = _silu_parts(a)
        h = silu * b
        do = g[:, None] * dys[ts]
        dh = do @ ew["w_down"]
        da, db = dh * b * d1, dh * silu
        E_do, E_h, E_a, E_b = u * np.abs(do), u * np.abs(h), u * np.abs(a), u * np.abs(b)
        E_dh = E_do @ np.abs(ew["w_down"])
        E_da = (u * np.abs(da) + np.abs(b * d1) * E_dh + np.abs(dh * b * d2) * E_a +
                np.abs(dh * d1) * E_b)
        E_db = u * np.abs(db) + np.abs(silu) * E_dh + np.abs(dh * d1) * E_a
        if e in ref["dw"]:
            bounds["dw_down"][e] = E_do.T @ np.abs(h) + np.abs(do).T @ E_h
            bounds["dw_gate"][e] = E_da.T @ np.abs(xe)
            bounds["dw_up"][e] = E_db.T @ np.abs(xe)
        E_dxp = E_da @ np.abs(ew["w_gate"]) + E_db @ np.abs(ew["w_up"])
        E_o = E_h @ np.abs(ew["w_down"]).T
        for r, (t, k) in enumerate(rows):
            if t in tok_pos:
                E_dxp_tok[tok_pos[t]] += E_dxp[r]
            if k >= 0:
                E_dg[t, k] = np.abs(dys[t]) @ E_o[r]
    if cfg.gate_mode == "renorm":
        sg = np.sum(gate * E_dg, axis=1, keepdims=True)
        E_dl = np.zeros((T, N))
        np.add.at(E_dl, (np.broadcast_to(np.arange(T)[:, None], idx.shape), idx),
                  gate * (E_dg + sg))
    else:
        E_dp = np.zeros((T, N))
        np.add.at(E_dp, (np.broadcast_to(np.arange(T)[:, None], idx.shape), idx), E_dg)
        E_dl = p * (E_dp + np.sum(p * E_dp, axis=1, keepdims=True))
    for e, dw in ref["dw"].items():  # experts without a kept row: exact zeros
        for k, v in dw.items():
            bounds.setdefault(k, {}).setdefault(e, np.zeros_like(v))
    w_r = O.f64(inp["w_r"])
    bounds["dx"] = E_dxp_tok + E_dl[tok] @ np.abs(w_r)
    if all_rows:
        bounds["dw_r"] = E_dl.T @ np.abs(xs)
        bounds["db_r"] = E_dl.sum(axis=0)
    return bounds


def run_backward(cfg: moe.LayerConfig, inp: dict, dy, z_coef: float, on_device: bool = False):
    """Forward (keeping state) then backward through the C ABI; returns the
    gradients (host copies, or the device tensors with on_device), the GPU
    routing (from moe_route, the same kernels), the forward's y and the
    statistics."""
    cfg = moe.LayerConfig(**{**cfg.__dict__, "save_for_backward": True})
    layer = moe.MoELayer(cfg, inp["w_r"], inp["b_r"], inp["experts"])
    y = layer.forward(inp["x"]).clone()
    g = layer.backward(dy, z_coef)
    torch.cuda.synchronize()
    st = layer.stats.to_host()
    T, K = cfg.T, cfg.top_k
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    gate = torch.zeros((T, K), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, inp["x"], inp["w_r"], inp["b_r"], idx, gate, None,
                  moe.alloc_workspace(cfg))
    torch.cuda.synchronize()
    out = dict(g) if on_device else {k: (None if v is None else v.cpu()) for k, v in g.items()}
    return out, idx.cpu().numpy().astype(np.int64), y.cpu(), st


def compare(name: str, got, ref: np.ndarray, bound=None) -> float:
    """bound None: max |err| <= GRAD_TOL_F32 * rms(ref); else elementwise
    |err| <= bound + 1e-3 * rms(ref). Returns max |err| / rms(ref)."""
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(got - ref)
    emax = float(err.max())
    if rms == 0.0:
        assert emax == 0.0, (name, emax)
        return 0.0
    if bound is None:
        assert emax <= GRAD_TOL_F32 * rms, (name, emax, rms, emax / rms)
    else:
        excess = err - (bound + 1e-3 * rms)
        assert excess.max() <= 0.0, (name, emax, rms, float(excess.max()))
    return emax / rms


def check_backward(cfg: moe.LayerConfig, inp: dict, dy, z_coef: float, *, tokens=None,
                   experts=None, router_grads: bool = True) -> dict:
    """GPU gradients against the float64 backward oracle on the GPU's routing
    (checked first, as in the forward tests). tokens / experts: the dx rows
    and expert weight gradients compared (None = all). fp32 layers: max |err|
    <= 1e-4 rms; bf16 (SwiGLU) layers: the per-element rounding bound of
    grad_rounding_bounds. Returns the ratios max |err| / rms per gradient."""
    grads, idx, _, st = run_backward(cfg, inp, dy, z_coef, on_device=True)
    assert st["status"] == 0
    K = cfg.top_k
    x, w_r = inp["x"].cpu(), inp["w_r"].cpu()
    b_r = None if inp["b_r"] is None else inp["b_r"].cpu()
    sb = None if cfg.select_bias is None else cfg.select_bias.cpu()
    l64 = O.router_logits(x, w_r, b_r)
    key64 = l64 if sb is None else l64 + O.f64(sb)[None, :]
    check_routing(key64, idx, K)
    ref = OG.moe_backward(x, w_r, b_r, expert_reader(inp["experts"]), dy.cpu(), K=K,
                          activation=cfg.activation, capacity_factor=stored_cf(cfg),
                          alpha=cfg.alpha, z_coef=z_coef, add_residual=cfg.add_residual,
                          gate_mode=cfg.gate_mode, select_bias=sb, n_shared=cfg.n_shared,
                          idx_override=idx, tokens=tokens, experts=experts,
                          router_grads=router_grads)
    bnd = None
    if cfg.dtype == "bf16":
        assert cfg.activation == "swiglu"
        bnd = grad_rounding_bounds(cfg, inp, dy.cpu(), ref)
    pick = (lambda k, e=None: None) if bnd is None else (
        lambda k, e=None: bnd[k] if e is None else bnd[k][e])
    ratios = {}
    tok = ref["tokens"]
    host = lambda t: t.cpu().numpy()  # copy only the compared slices off the device
    ratios["dx"] = compare("dx", host(grads["dx"][torch.as_tensor(tok, device="cuda")]),
                           ref["dx"], pick("dx"))
    if router_grads:
        ratios["dw_r"] = compare("dw_r", host(grads["dw_r"]), ref["dw_r"], pick("dw_r"))
        if b_r is not None:
            ratios["db_r"] = compare("db_r", host(grads["db_r"]), ref["db_r"], pick("db_r"))
    for e, dw in ref["dw"].items():
        for k, v in dw.items():
            r = compare(f"{k}[{e}]", host(grads[k][e]), v, pick(k, e))
            ratios[k] = max(ratios.get(k, 0.0), r)
    return ratios
