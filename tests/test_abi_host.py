"""Host-side checks of the C ABI (no GPU): the library builds and loads, it
exports every function include/moe.h declares, and the host logic (argument
checks, capacity, workspace size, path choice) behaves as declared. Only
calls that return before any launch are made here."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import mixture_experts_layer_101_b300 as moe
from mixture_experts_layer_101_b300 import build as moe_build
from mixture_experts_layer_101_b300 import moe as M
from oracle import moe_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        moe_build.build()
    return moe.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(moe.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def cfg(**kw):
    base = dict(T=4096, d_model=4096, d_ff=14336, n_experts=8, top_k=2)
    base.update(kw)
    return moe.LayerConfig(**base)


def test_capacity_matches_oracle(lib):
    for K, N, T in [(1, 64, 32768), (2, 8, 512), (3, 7, 1000), (8, 256, 4096), (1, 1, 1)]:
        for cf in np.float32([0.01, 0.1, 0.7, 1.0, 1.25, 1.3333, 2.0]):
            c = cfg(T=T, n_experts=N, top_k=K, capacity_factor=float(cf))
            assert moe.capacity(c) == O.capacity(K, N, float(cf), T)
    assert moe.capacity(cfg(capacity_factor=math.inf)) == 2 ** 31 - 1
    assert moe.capacity(cfg(capacity_factor=0.0)) == 2 ** 31 - 1
    assert moe.capacity(cfg(capacity_factor=-2.0)) == 2 ** 31 - 1


def test_workspace_size(lib):
    c = cfg()
    A = 4096 * 2
    n = moe.workspace_size(c)
    assert n >= A * 4096 * 2 + A * 14336 * 2 + A * 4096 * 4
    assert n % 256 == 0
    # capacity bounds the slot count
    small = cfg(capacity_factor=0.5)
    assert moe.a_max(small) == 8 * 512 and moe.workspace_size(small) < n
    assert moe.workspace_size(cfg(top_k=9, n_experts=16)) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(top_k=3, n_experts=2), M.MOE_ERR_INVALID),
    (dict(top_k=0), M.MOE_ERR_INVALID),
    (dict(T=-1), M.MOE_ERR_INVALID),
    (dict(capacity_factor=math.nan), M.MOE_ERR_INVALID),
    (dict(n_experts=300), M.MOE_ERR_UNSUPPORTED),
    (dict(top_k=9, n_experts=16), M.MOE_ERR_UNSUPPORTED),
    (dict(T=(1 << 24) + 1), M.MOE_ERR_UNSUPPORTED),
    (dict(d_model=4092), M.MOE_ERR_UNSUPPORTED),
    (dict(has_bias=True), M.MOE_ERR_UNSUPPORTED),
])
def test_invalid_configs_are_rejected_before_launch(lib, kw, code):
    c = cfg(**kw).c()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the call fails first
    w = M.MoEExpertWeightsC(fake, fake, fake, None, None, None, None)
    r = lib.moe_forward(ctypes.byref(c), fake, fake, None, ctypes.byref(w), fake, None, fake, None)
    assert r == code
    r = lib.moe_route(ctypes.byref(c), fake, fake, None, fake, fake, None, fake, None)
    assert r == code


def test_bad_pointers_are_rejected_before_launch(lib):
    c = cfg().c()
    ok = ctypes.c_void_p(1 << 20)
    w = M.MoEExpertWeightsC(ok, ok, ok, None, None, None, None)
    assert lib.moe_forward(ctypes.byref(c), None, ok, None, ctypes.byref(w), ok, None, ok,
                           None) == M.MOE_ERR_INVALID
    mis = ctypes.c_void_p((1 << 20) + 8)
    assert lib.moe_forward(ctypes.byref(c), mis, ok, None, ctypes.byref(w), ok, None, ok,
                           None) == M.MOE_ERR_INVALID
    assert lib.moe_forward(ctypes.byref(c), ok, ok, None, ctypes.byref(w), ok, None, None,
                           None) == M.MOE_ERR_WORKSPACE
    ws_mis = ctypes.c_void_p((1 << 20) + 128)
    assert lib.moe_forward(ctypes.byref(c), ok, ok, None, ctypes.byref(w), ok, None, ws_mis,
                           None) == M.MOE_ERR_WORKSPACE
    w_missing = M.MoEExpertWeightsC(ok, None, ok, None, None, None, None)
    assert lib.moe_forward(ctypes.byref(c), ok, ok, None, ctypes.byref(w_missing), ok, None, ok,
                           None) == M.MOE_ERR_INVALID
    g = cfg(activation="gelu", has_bias=True, dtype="f32").c()
    w_nobias = M.MoEExpertWeightsC(None, None, None, ok, None, ok, None)
    assert lib.moe_expert_ffn(ctypes.byref(g), ok, ok, ctypes.byref(w_nobias), ok, None, ok,
                              None) == M.MOE_ERR_INVALID
    assert lib.moe_combine(ctypes.byref(cfg(add_residual=True).c()), ok, ok, ok, None, ok,
                           None) == M.MOE_ERR_INVALID


def test_status_strings(lib):
    for code in range(8):
        s = moe.status_string(code)
        assert s and s != "unknown status"
    assert moe.status_string(99) == "unknown status"


def test_launch_count(lib):
    # router (tensor cores: weight split, GEMM, top-K; fused: split, GEMM;
    # CUDA cores, or T <= 128 with N <= 32: one kernel), statistics (one block
    # while every row has at most 64 partial blocks, else per-row reduction +
    # L_aux), dispatch (4; at most 256 tokens: 2), the two expert GEMMs, the
    # combine
    assert moe.forward_launch_count(cfg()) == 12          # tensor-core router
    assert moe.forward_launch_count(cfg(dtype="f32")) == 10
    assert moe.forward_launch_count(cfg(d_model=72)) == 10  # d % 64 != 0: CUDA-core router
    assert moe.forward_launch_count(cfg(top_k=9, n_experts=16)) == -1
    # one K split and one expert tile: selection runs in the router GEMM epilogue
    assert moe.forward_launch_count(cfg(T=32768, d_model=1024, n_experts=64, top_k=1)) == 11
    # small-batch router: one block and one statistics partial per token
    assert moe.forward_launch_count(cfg(T=100, d_model=64)) == 8  # 100 partials: two kernels
    assert moe.forward_launch_count(cfg(T=64, d_model=64)) == 7   # 64 partials: one block
    assert moe.forward_launch_count(cfg(T=4096, n_experts=256, top_k=8)) == 12  # two tiles
    # decode: the small-batch router, 16 partials (one statistics kernel); the
    # split gate/up reduction adds its SwiGLU pass
    assert moe.forward_launch_count(cfg(T=16)) == 8
    assert moe.forward_launch_count(cfg(T=1 << 24, d_model=64, n_experts=8, top_k=2)) == 11


def test_tensor_core_path_choice(lib):
    assert moe.ffn_uses_tensor_cores(cfg())
    assert moe.ffn_uses_tensor_cores(cfg(d_model=7168, d_ff=2048, n_experts=256, top_k=8))
    assert moe.ffn_uses_tensor_cores(cfg(d_model=1024, d_ff=4096, n_experts=64, top_k=1))
    assert not moe.ffn_uses_tensor_cores(cfg(dtype="f32"))
    assert not moe.ffn_uses_tensor_cores(cfg(d_model=72))
    assert not moe.ffn_uses_tensor_cores(cfg(d_ff=100))
    assert not moe.ffn_uses_tensor_cores(cfg(activation="gelu"))


def test_binding_refuses_cpu_tensors(lib):
    import torch
    c = cfg(T=4, d_model=256, d_ff=128, n_experts=4)
    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        moe.moe_combine(c, x, x, x, x, x)
