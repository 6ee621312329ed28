"""Seeded synthetic inputs for the sparse-MoE forward layer.

This module only draws random numbers and names workloads. It holds none of
the layer's arithmetic, so both the CUDA path and the float64 oracle can take
their inputs from here (the oracle reads back exactly the stored tensors).

Workloads (shapes and distributions of the layers the MoE pages discuss):

  tiny_fp32        T=64 (1x64), d=64, N=4, K=2, GELU experts 64->128->64 with
                   bias, router Linear(64->4) with bias; x ~ N(0,1); every
                   weight and bias ~ U(+-1/sqrt(fan_in)); no capacity limit.
  mixtral_prefill  T=4096 (2x2048), d=4096, N=8, K=2, SwiGLU F=14336, no bias,
                   router 4096->8 fp32; x ~ N(0,1); weights ~ N(0, 0.02).
  mixtral_decode   T=16, same weights and shapes as mixtral_prefill.
  deepseek_fine    T=4096, d=7168, N=256, K=8, SwiGLU F=2048, router
                   7168->256 fp32; x ~ N(0,1); weights ~ N(0, 0.02).
  deepseek_shared  deepseek_fine plus one shared expert (F=2048) on every
                   token (the fine-grained + shared layout of DeepSeek-MoE).
  switch_skewed    T=32768 (16x2048), d=1024, N=64, K=1, SwiGLU F=4096,
                   CF=1.25 (capacity 640), residual on; router bias
                   SWITCH_SKEW_BIAS on experts 0..3 so that about 70% of the
                   tokens prefer those four experts.

Seeds: x uses seed 0, expert e uses seed 1 + e, the router uses seed 1000,
the output gradient dy of the backward pass seed 2000.
Values are drawn in fp32 and then cast to the storage dtype. x and the router
are always drawn on the CPU generator (so they are identical on every
machine); expert weights are drawn on the device they are created on.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

# Router bias for switch_skewed, added to experts 0..3. Derived by
# oracle/calibrate_switch_bias.py (bisection with the float64 oracle on the
# seed-0 x and router weights of switch_skewed): 70.2% of the 32768 tokens
# then have their largest logit on experts 0..3.
SWITCH_SKEW_BIAS = 1.109375
SWITCH_SKEW_EXPERTS = 4

X_SEED = 0
ROUTER_SEED = 1000
SELECT_BIAS_SEED = 1001
DY_SEED = 2000


def expert_seed(e: int) -> int:
    return 1 + e


@dataclass(frozen=True)
class MoEWorkload:
    name: str
    T: int
    d: int
    F: int
    N: int
    K: int
    dtype: str = "bf16"          # "bf16" | "f32": x, expert weights, y
    activation: str = "swiglu"   # "swiglu" | "gelu"
    has_bias: bool = False       # expert biases (GELU experts only)
    router_bias: str = "none"    # "none" | "uniform" | "skew"
    capacity_factor: float = math.inf
    alpha: float = 0.01
    add_residual: bool = False
    init: str = "normal"         # "normal" (std w_std) | "uniform" (1/sqrt(fan_in))
    w_std: float = 0.02
    router_std: float = 0.02
    gate_mode: str = "renorm"    # "renorm" | "softmax"
    select_bias: str = "none"    # "none" | "uniform": a top-K selection bias
    n_shared: int = 0            # shared experts, seeds 1 + N + s after the routed ones

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


WORKLOADS = {
    "tiny_fp32": MoEWorkload("tiny_fp32", T=64, d=64, F=128, N=4, K=2, dtype="f32",
                             activation="gelu", has_bias=True, router_bias="uniform",
                             init="uniform"),
    "mixtral_prefill": MoEWorkload("mixtral_prefill", T=4096, d=4096, F=14336, N=8, K=2),
    "mixtral_decode": MoEWorkload("mixtral_decode", T=16, d=4096, F=14336, N=8, K=2),
    "deepseek_fine": MoEWorkload("deepseek_fine", T=4096, d=7168, F=2048, N=256, K=8),
    "deepseek_shared": MoEWorkload("deepseek_shared", T=4096, d=7168, F=2048, N=256, K=8,
                                   n_shared=1),
    "switch_skewed": MoEWorkload("switch_skewed", T=32768, d=1024, F=4096, N=64, K=1,
                                 router_bias="skew", capacity_factor=1.25,
                                 add_residual=True),
}

# Order in which the workloads are listed; the first is the small case.
WORKLOAD_ORDER = ["tiny_fp32", "mixtral_prefill", "mixtral_decode", "deepseek_fine",
                  "switch_skewed"]


def workload(name: str, **overrides) -> MoEWorkload:
    return replace(WORKLOADS[name], **overrides)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _uniform(shape, bound, gen, device):
    return (torch.rand(shape, generator=gen, device=device, dtype=torch.float32) * 2 - 1) * bound


def make_x(w: MoEWorkload, T: int | None = None, device="cpu") -> torch.Tensor:
    """x [T][d] in the storage dtype, N(0, 1), seed 0, drawn on `device` (the
    CPU and CUDA generators give different numbers for the same seed: the
    very large cases draw on the GPU, and the oracle then reads x back)."""
    T = w.T if T is None else T
    g = _gen(X_SEED, device)
    return torch.randn((T, w.d), generator=g, device=device,
                       dtype=torch.float32).to(w.torch_dtype)


def make_dy(w: MoEWorkload, T: int | None = None) -> torch.Tensor:
    """Output gradient dy [T][d] for the backward pass on the CPU: N(0, 1) in
    the storage dtype, seed 2000."""
    T = w.T if T is None else T
    g = _gen(DY_SEED, "cpu")
    return torch.randn((T, w.d), generator=g, dtype=torch.float32).to(w.torch_dtype)


def make_router(w: MoEWorkload, skew_bias: float | None = None):
    """(w_r [N][d] fp32, b_r [N] fp32 or None) on the CPU."""
    g = _gen(ROUTER_SEED, "cpu")
    if w.init == "uniform":
        bound = 1.0 / math.sqrt(w.d)
        w_r = _uniform((w.N, w.d), bound, g, "cpu")
    else:
        w_r = torch.randn((w.N, w.d), generator=g, dtype=torch.float32) * w.router_std
    b_r = None
    if w.router_bias == "uniform":
        b_r = _uniform((w.N,), 1.0 / math.sqrt(w.d), g, "cpu")
    elif w.router_bias == "skew":
        beta = SWITCH_SKEW_BIAS if skew_bias is None else skew_bias
        b_r = torch.zeros(w.N, dtype=torch.float32)
        b_r[:SWITCH_SKEW_EXPERTS] = beta
    return w_r.contiguous(), (None if b_r is None else b_r.contiguous())


def make_select_bias(w: MoEWorkload):
    """Top-K selection bias [N] fp32 on the CPU (None unless requested):
    U(-0.5, 0.5), seed 1001."""
    if w.select_bias == "none":
        return None
    g = _gen(SELECT_BIAS_SEED, "cpu")
    return _uniform((w.N,), 0.5, g, "cpu").contiguous()


def make_expert(w: MoEWorkload, e: int, device="cpu") -> dict:
    """Weights of expert e (nn.Linear (out, in) layout) in the storage dtype."""
    g = _gen(expert_seed(e), device)
    dt = w.torch_dtype
    if w.activation == "swiglu":
        def mat(rows, cols):
            if w.init == "uniform":
                return _uniform((rows, cols), 1.0 / math.sqrt(cols), g, device)
            return torch.randn((rows, cols), generator=g, device=device,
                               dtype=torch.float32) * w.w_std
        wg = mat(w.F, w.d).to(dt)
        wu = mat(w.F, w.d).to(dt)
        wd = mat(w.d, w.F).to(dt)
        return {"w_gate": wg, "w_up": wu, "w_down": wd}
    # GELU expert: Linear(d -> F) + GELU + Linear(F -> d)
    if w.init == "uniform":
        w1 = _uniform((w.F, w.d), 1.0 / math.sqrt(w.d), g, device)
        b1 = _uniform((w.F,), 1.0 / math.sqrt(w.d), g, device)
        w2 = _uniform((w.d, w.F), 1.0 / math.sqrt(w.F), g, device)
        b2 = _uniform((w.d,), 1.0 / math.sqrt(w.F), g, device)
    else:
        w1 = torch.randn((w.F, w.d), generator=g, device=device) * w.w_std
        b1 = torch.randn((w.F,), generator=g, device=device) * w.w_std
        w2 = torch.randn((w.d, w.F), generator=g, device=device) * w.w_std
        b2 = torch.randn((w.d,), generator=g, device=device) * w.w_std
    out = {"w1": w1.to(dt), "w2": w2.to(dt)}
    if w.has_bias:
        out["b1"] = b1.to(dt)
        out["b2"] = b2.to(dt)
    return out


def make_experts(w: MoEWorkload, device="cpu") -> dict:
    """All expert weights stacked over experts, the N routed ones then the
    n_shared shared ones: [N + n_shared][...] in the storage dtype."""
    names = (["w_gate", "w_up", "w_down"] if w.activation == "swiglu"
             else (["w1", "b1", "w2", "b2"] if w.has_bias else ["w1", "w2"]))
    first = make_expert(w, 0, device)
    E = w.N + w.n_shared
    stacked = {k: torch.empty((E,) + tuple(first[k].shape), dtype=first[k].dtype,
                              device=device) for k in names}
    for e in range(E):
        ex = first if e == 0 else make_expert(w, e, device)
        for k in names:
            stacked[k][e].copy_(ex[k])
        del ex
    return stacked


def make_inputs(w: MoEWorkload, device="cpu") -> dict:
    """Every input of the layer: x, w_r, b_r and the stacked expert weights."""
    x = make_x(w)
    w_r, b_r = make_router(w)
    out = {"x": x.to(device), "w_r": w_r.to(device),
           "b_r": None if b_r is None else b_r.to(device)}
    out.update(make_experts(w, device))
    return out
