"""Python binding of libmoe (include/moe.h) over ctypes.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Tensors are torch CUDA tensors (device memory and streams come from
PyTorch); each function passes their device pointers and the current CUDA
stream to the C entry point of the same name and raises MoEError when the
status is not MOE_OK. There is no CPU path: without the built library or a
CUDA device every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3
MOE_ERR_TIMEOUT, MOE_ERR_NONFINITE, MOE_ERR_WORKSPACE, MOE_ERR_INDEX = 4, 5, 6, 7
MOE_F32, MOE_BF16 = 0, 1
MOE_SWIGLU, MOE_GELU = 0, 1
MOE_GATE_RENORM, MOE_GATE_SOFTMAX = 0, 1

# Every symbol the header declares, in declaration order.
EXPORTED = ["moe_workspace_size", "moe_capacity", "moe_route", "moe_route_no_workspace",
            "moe_dispatch",
            "moe_expert_ffn", "moe_combine", "moe_forward", "moe_status_string",
            "moe_backward", "moe_trace_events", "moe_selftest_bounded_wait",
            "moe_forward_launch_count", "moe_backward_launch_count",
            "moe_ffn_uses_tensor_cores", "moe_ep_workspace_size", "moe_ep_pack",
            "moe_ep_regroup", "moe_ep_regroup_back", "moe_ep_unpack"]


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


class MoEConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("activation", ctypes.c_int32),
                ("has_bias", ctypes.c_int32), ("capacity_factor", ctypes.c_float),
                ("alpha", ctypes.c_float), ("add_residual", ctypes.c_int32),
                ("gate_mode", ctypes.c_int32), ("select_bias", ctypes.c_void_p),
                ("n_shared", ctypes.c_int32), ("save_for_backward", ctypes.c_int32)]


class MoEStatsC(ctypes.Structure):
    _fields_ = [("count", ctypes.c_void_p), ("kept", ctypes.c_void_p),
                ("n_dropped", ctypes.c_void_p), ("f", ctypes.c_void_p), ("P", ctypes.c_void_p),
                ("l_aux", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("z_loss", ctypes.c_void_p), ("entropy", ctypes.c_void_p)]


class MoEExpertWeightsC(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("w1", ctypes.c_void_p), ("b1", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("b2", ctypes.c_void_p)]


class MoEGradsC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("dx", "dw_r", "db_r", "dw_gate", "dw_up",
                                               "dw_down", "dw1", "db1", "dw2", "db2")]


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libmoe.so: the in-tree build, or the file named by the environment
    variable MOE_LIBRARY (another build of the same sources, e.g. to compare
    two builds in one process tree); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("MOE_LIBRARY") or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe.so not found at {path}: build it with "
                           "`python -m mixture_experts_layer_101_b300.build`")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    cfgp = ctypes.POINTER(MoEConfig)
    statp = ctypes.POINTER(MoEStatsC)
    wp = ctypes.POINTER(MoEExpertWeightsC)
    lib.moe_workspace_size.argtypes = [cfgp]
    lib.moe_workspace_size.restype = ctypes.c_size_t
    lib.moe_capacity.argtypes = [cfgp]
    lib.moe_capacity.restype = ctypes.c_int32
    lib.moe_selftest_bounded_wait.argtypes = [ctypes.c_uint32, P, P]
    lib.moe_selftest_bounded_wait.restype = ctypes.c_int
    lib.moe_forward_launch_count.argtypes = [cfgp]
    lib.moe_forward_launch_count.restype = ctypes.c_int32
    lib.moe_ffn_uses_tensor_cores.argtypes = [cfgp]
    lib.moe_ffn_uses_tensor_cores.restype = ctypes.c_int32
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_route.argtypes = [cfgp, P, P, P, P, P, statp, P, P]
    lib.moe_route_no_workspace.argtypes = [cfgp, P, P, P, P, P, statp, P]
    lib.moe_route_no_workspace.restype = ctypes.c_int
    lib.moe_dispatch.argtypes = [cfgp, P, P, P, P, P, P, statp, P, P]
    lib.moe_expert_ffn.argtypes = [cfgp, P, P, wp, P, statp, P, P]
    lib.moe_combine.argtypes = [cfgp, P, P, P, P, P, P]
    lib.moe_forward.argtypes = [cfgp, P, P, P, wp, P, statp, P, P]
    lib.moe_backward.argtypes = [cfgp, P, P, wp, P, ctypes.c_float,
                                 ctypes.POINTER(MoEGradsC), statp, P, P]
    lib.moe_backward_launch_count.argtypes = [cfgp]
    lib.moe_backward_launch_count.restype = ctypes.c_int32
    lib.moe_trace_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32]
    lib.moe_trace_events.restype = ctypes.c_int
    lib.moe_ep_workspace_size.argtypes = [cfgp, ctypes.c_int32]
    lib.moe_ep_workspace_size.restype = ctypes.c_size_t
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.moe_ep_pack.argtypes = [cfgp, i32, P, P, P, P, P, statp, P, P]
    lib.moe_ep_regroup.argtypes = [cfgp, i32, i32, P, P, i64, P, P, P, statp, P, P]
    lib.moe_ep_regroup_back.argtypes = [cfgp, i32, i32, P, P, i64, P, P, statp, P, P]
    lib.moe_ep_unpack.argtypes = [cfgp, i32, P, P, P, P, statp, P, P]
    for name in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward",
                 "moe_backward", "moe_ep_pack", "moe_ep_regroup", "moe_ep_regroup_back",
                 "moe_ep_unpack"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().moe_status_string(int(code)).decode()


moe_status_string = status_string


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
@dataclass
class LayerConfig:
    T: int
    d_model: int
    d_ff: int
    n_experts: int
    top_k: int
    dtype: str = "bf16"
    activation: str = "swiglu"
    has_bias: bool = False
    capacity_factor: float = math.inf
    alpha: float = 0.01
    add_residual: bool = False
    gate_mode: str = "renorm"          # "renorm" | "softmax"
    select_bias: torch.Tensor | None = None  # [N] fp32 CUDA tensor: top-K choice only
    n_shared: int = 0                  # shared experts after the N routed ones
    save_for_backward: bool = False    # forward keeps what moe_backward needs

    @classmethod
    def from_workload(cls, w, T: int | None = None) -> "LayerConfig":
        return cls(T=w.T if T is None else T, d_model=w.d, d_ff=w.F, n_experts=w.N, top_k=w.K,
                   dtype=w.dtype, activation=w.activation, has_bias=w.has_bias,
                   capacity_factor=w.capacity_factor, alpha=w.alpha, add_residual=w.add_residual,
                   gate_mode=getattr(w, "gate_mode", "renorm"),
                   n_shared=getattr(w, "n_shared", 0))

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def c(self) -> MoEConfig:
        return MoEConfig(self.T, self.d_model, self.d_ff, self.n_experts, self.top_k,
                         MOE_BF16 if self.dtype == "bf16" else MOE_F32,
                         MOE_SWIGLU if self.activation == "swiglu" else MOE_GELU,
                         int(self.has_bias), float(self.capacity_factor), float(self.alpha),
                         int(self.add_residual),
                         MOE_GATE_SOFTMAX if self.gate_mode == "softmax" else MOE_GATE_RENORM,
                         _ptr(self.select_bias), int(self.n_shared),
                         int(self.save_for_backward))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("libmoe takes CUDA tensors only (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoEError(code, where)


class Stats:
    """Device tensors for the layer statistics (count, kept, n_dropped, f, P,
    l_aux, status)."""

    def __init__(self, n_experts: int, device="cuda"):
        i32, f32 = torch.int32, torch.float32
        self.count = torch.zeros(n_experts, dtype=i32, device=device)
        self.kept = torch.zeros(n_experts, dtype=i32, device=device)
        self.n_dropped = torch.zeros(1, dtype=i32, device=device)
        self.f = torch.zeros(n_experts, dtype=f32, device=device)
        self.P = torch.zeros(n_experts, dtype=f32, device=device)
        self.l_aux = torch.zeros(1, dtype=f32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.z_loss = torch.zeros(1, dtype=f32, device=device)
        self.entropy = torch.zeros(1, dtype=f32, device=device)

    def c(self) -> MoEStatsC:
        return MoEStatsC(*(_ptr(t) for t in (self.count, self.kept, self.n_dropped, self.f,
                                             self.P, self.l_aux, self.status, self.z_loss,
                                             self.entropy)))

    def status_bits(self) -> int:
        return int(self.status.item()) & 0xFFFFFFFF

    def to_host(self) -> dict:
        return {"count": self.count.cpu().numpy(), "kept": self.kept.cpu().numpy(),
                "n_dropped": int(self.n_dropped.item()), "f": self.f.cpu().numpy(),
                "P": self.P.cpu().numpy(), "l_aux": float(self.l_aux.item()),
                "status": self.status_bits(), "z_loss": float(self.z_loss.item()),
                "entropy": float(self.entropy.item())}


def weights_c(weights: dict) -> MoEExpertWeightsC:
    names = ("w_gate", "w_up", "w_down", "w1", "b1", "w2", "b2")
    return MoEExpertWeightsC(*(_ptr(weights.get(n)) for n in names))


def workspace_size(cfg: LayerConfig) -> int:
    return int(load_library().moe_workspace_size(ctypes.byref(cfg.c())))


moe_workspace_size = workspace_size


def capacity(cfg: LayerConfig) -> int:
    return int(load_library().moe_capacity(ctypes.byref(cfg.c())))


moe_capacity = capacity


def ffn_uses_tensor_cores(cfg: LayerConfig) -> bool:
    return load_library().moe_ffn_uses_tensor_cores(ctypes.byref(cfg.c())) == 1


moe_ffn_uses_tensor_cores = ffn_uses_tensor_cores


def backward_launch_count(cfg: LayerConfig) -> int:
    """Kernels one moe_backward launches for cfg (db_r requested); -1 if cfg
    does not save for backward."""
    return int(load_library().moe_backward_launch_count(ctypes.byref(cfg.c())))


moe_backward_launch_count = backward_launch_count


def forward_launch_count(cfg: LayerConfig) -> int:
    """Kernels one moe_forward launches for cfg (all statistics requested)."""
    return int(load_library().moe_forward_launch_count(ctypes.byref(cfg.c())))


moe_forward_launch_count = forward_launch_count


def a_max(cfg: LayerConfig) -> int:
    """Most routed assignments capacity lets through: min(T*K, N*C)."""
    C = capacity(cfg)
    return min(cfg.T * cfg.top_k, cfg.n_experts * C)


def rows_max(cfg: LayerConfig) -> int:
    """Rows of the permuted buffers (x_perm, h, o): routed A_max + shared S*T."""
    return a_max(cfg) + cfg.n_shared * cfg.T


def alloc_workspace(cfg: LayerConfig, device="cuda") -> torch.Tensor:
    """A byte tensor of moe_workspace_size(cfg) bytes (torch allocations are
    at least 256-byte aligned)."""
    n = workspace_size(cfg)
    if n == 0:
        raise MoEError(MOE_ERR_INVALID, "moe_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


# --------------------------------------------------------------------------
# the C entry points, one by one
# --------------------------------------------------------------------------
def moe_route(cfg: LayerConfig, x, w_r, b_r, idx, gate, stats: Stats | None, ws, stream=None):
    lib = load_library()
    st = stats.c() if stats is not None else None
    code = lib.moe_route(ctypes.byref(cfg.c()), _ptr(x), _ptr(w_r), _ptr(b_r), _ptr(idx),
                         _ptr(gate), ctypes.byref(st) if st is not None else None, _ptr(ws),
                         _stream(stream))
    _check(code, "moe_route")


def moe_route_no_workspace(cfg: LayerConfig, x, w_r, b_r, idx, gate, stats: Stats | None,
                           stream=None):
    """moe_route without a workspace: for callers that cannot allocate device
    memory. It always runs a CUDA-core router (moe_route takes the tensor-
    core router for bf16 layers with d % 64 == 0 beyond 128 tokens or 32
    experts, so the two can choose differently on near-tie tokens; below
    that both run the small-batch router). The library keeps the statistics'
    partial sums in a fixed 1 MiB array (ceil(T/32) * (N + 2) <= 131072,
    else MOE_ERR_WORKSPACE); calls share it, so calls that overlap on the GPU
    must not be issued. The first call in a CUDA context (normally once per
    device) looks up the array's address; make it before any stream
    capture."""
    lib = load_library()
    st = stats.c() if stats is not None else None
    code = lib.moe_route_no_workspace(ctypes.byref(cfg.c()), _ptr(x), _ptr(w_r), _ptr(b_r),
                                      _ptr(idx), _ptr(gate),
                                      ctypes.byref(st) if st is not None else None,
                                      _stream(stream))
    _check(code, "moe_route_no_workspace")


def moe_dispatch(cfg: LayerConfig, x, idx, offsets, slot_of, token_of_slot, x_perm,
                 stats: Stats | None, ws, stream=None):
    lib = load_library()
    st = stats.c() if stats is not None else None
    code = lib.moe_dispatch(ctypes.byref(cfg.c()), _ptr(x), _ptr(idx), _ptr(offsets),
                            _ptr(slot_of), _ptr(token_of_slot), _ptr(x_perm),
                            ctypes.byref(st) if st is not None else None, _ptr(ws),
                            _stream(stream))
    _check(code, "moe_dispatch")


def moe_expert_ffn(cfg: LayerConfig, x_perm, offsets, weights: dict, o, stats: Stats | None, ws,
                   stream=None):
    lib = load_library()
    st = stats.c() if stats is not None else None
    wc = weights_c(weights)
    code = lib.moe_expert_ffn(ctypes.byref(cfg.c()), _ptr(x_perm), _ptr(offsets),
                              ctypes.byref(wc), _ptr(o),
                              ctypes.byref(st) if st is not None else None, _ptr(ws),
                              _stream(stream))
    _check(code, "moe_expert_ffn")


def moe_combine(cfg: LayerConfig, o, slot_of, gate, x, y, stream=None):
    lib = load_library()
    code = lib.moe_combine(ctypes.byref(cfg.c()), _ptr(o), _ptr(slot_of), _ptr(gate), _ptr(x),
                           _ptr(y), _stream(stream))
    _check(code, "moe_combine")


def moe_forward(cfg: LayerConfig, x, w_r, b_r, weights: dict, y, stats: Stats | None, ws,
                stream=None):
    lib = load_library()
    st = stats.c() if stats is not None else None
    wc = weights_c(weights)
    code = lib.moe_forward(ctypes.byref(cfg.c()), _ptr(x), _ptr(w_r), _ptr(b_r),
                           ctypes.byref(wc), _ptr(y), ctypes.byref(st) if st is not None else None,
                           _ptr(ws), _stream(stream))
    _check(code, "moe_forward")


GRAD_NAMES = ("dx", "dw_r", "db_r", "dw_gate", "dw_up", "dw_down", "dw1", "db1", "dw2", "db2")


def grads_c(grads: dict) -> MoEGradsC:
    return MoEGradsC(*(_ptr(grads.get(n)) for n in GRAD_NAMES))


def alloc_grads(cfg: LayerConfig, router_bias: bool = True, device="cuda") -> dict:
    """fp32 gradient buffers shaped like the inputs and weights they belong to."""
    T, d, F, N = cfg.T, cfg.d_model, cfg.d_ff, cfg.n_experts
    E = N + cfg.n_shared
    z = lambda *shape: torch.empty(shape, dtype=torch.float32, device=device)
    g = {"dx": z(T, d), "dw_r": z(N, d), "db_r": z(N) if router_bias else None}
    if cfg.activation == "swiglu":
        g.update(dw_gate=z(E, F, d), dw_up=z(E, F, d), dw_down=z(E, d, F))
    else:
        g.update(dw1=z(E, F, d), dw2=z(E, d, F))
        if cfg.has_bias:
            g.update(db1=z(E, F), db2=z(E, d))
    return g


def moe_backward(cfg: LayerConfig, x, w_r, weights: dict, dy, z_coef: float, grads: dict,
                 stats: Stats | None, ws, stream=None):
    lib = load_library()
    _check(lib.moe_backward(ctypes.byref(cfg.c()), _ptr(x), _ptr(w_r),
                            ctypes.byref(weights_c(weights)), _ptr(dy), float(z_coef),
                            ctypes.byref(grads_c(grads)),
                            ctypes.byref(stats.c()) if stats else None, _ptr(ws),
                            _stream(stream)), "moe_backward")


def moe_trace_events(events):
    """Register up to 8 raw CUDA event handles (ints, e.g. TraceEvents.handles)
    that moe_forward / moe_backward record at their stage boundaries on this
    host thread; pass [] to clear. The caller keeps the events alive while
    registered."""
    lib = load_library()
    arr = (ctypes.c_void_p * max(len(events), 1))(*[ctypes.c_void_p(int(e)) for e in events])
    _check(lib.moe_trace_events(arr if events else None, len(events)), "moe_trace_events")


class TraceEvents:
    """A set of raw CUDA events for moe_trace_events, created and timed with
    the CUDA runtime bindings (torch.cuda.Event cannot time events that it
    did not record itself)."""

    def __init__(self, n: int = 6):
        from cuda.bindings import runtime as rt
        self._rt = rt
        self.events = []
        for _ in range(n):
            err, ev = rt.cudaEventCreate()
            if err != rt.cudaError_t.cudaSuccess:
                raise RuntimeError(f"cudaEventCreate failed: {err}")
            self.events.append(ev)

    def handles(self):
        return [int(e) for e in self.events]

    def elapsed_ms(self, i: int, j: int) -> float:
        err, ms = self._rt.cudaEventElapsedTime(self.events[i], self.events[j])
        if err != self._rt.cudaError_t.cudaSuccess:
            raise RuntimeError(f"cudaEventElapsedTime failed: {err}")
        return float(ms)

    def close(self):
        for e in self.events:
            self._rt.cudaEventDestroy(e)
        self.events = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_selftest_bounded_wait(limit_us: int, status, stream=None):
    """Runs the bounded-wait self-test: a device wait that nothing satisfies
    gives up after limit_us and sets the MOE_ERR_TIMEOUT bit in status (an
    int32 CUDA tensor)."""
    lib = load_library()
    _check(lib.moe_selftest_bounded_wait(int(limit_us), _ptr(status), _stream(stream)),
           "moe_selftest_bounded_wait")


TRACE_STAGES = ["router", "dispatch", "ffn_gate_up", "ffn_down", "combine"]
# intervals between moe_backward's eight trace events
TRACE_STAGES_BWD = ["bwd_combine_router", "bwd_down_dgrad", "bwd_down_wgrad",
                    "bwd_gate_up_dgrad", "bwd_gate_up_wgrad", "bwd_dx", "bwd_router_wgrad"]


def capture_graph(fn, device=None) -> "torch.cuda.CUDAGraph":
    """Runs fn() (a sequence of library calls on the current stream) once
    eagerly, so that the library's one-time per-device setup (kernel
    attributes, the CUDA driver's tensor-map encoder) stays out of the capture,
    then records fn() as a CUDA graph; graph.replay() runs the same kernels
    with the same arguments again. Trace events registered while fn runs
    (moe_trace_events) are recorded into the graph too."""
    fn()
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


class MoELayer:
    """A sparse-MoE FFN layer with its weights, workspace and statistics held
    on one CUDA device; forward() runs moe_forward."""

    def __init__(self, cfg: LayerConfig, w_r, b_r, weights: dict, device="cuda"):
        self.cfg = cfg
        self.w_r = w_r
        self.b_r = b_r
        self.weights = weights
        self.ws = alloc_workspace(cfg, device)
        self.stats = Stats(cfg.n_experts, device)
        self.y = torch.empty((cfg.T, cfg.d_model), dtype=cfg.torch_dtype, device=device)

    def forward(self, x, stream=None):
        moe_forward(self.cfg, x, self.w_r, self.b_r, self.weights, self.y, self.stats, self.ws,
                    stream)
        self._x = x
        return self.y

    def capture(self, x) -> "torch.cuda.CUDAGraph":
        """Records one forward() on the input buffer x as a CUDA graph: the
        layer's kernels with their arguments, captured once, so that a decode
        loop replays them (graph.replay()) without a launch per kernel. A
        replay reads what x holds at that time and writes self.y and
        self.stats; x, the weights and the workspace must stay where they
        are."""
        return capture_graph(lambda: self.forward(x), self.ws.device)

    def backward(self, dy, z_coef: float = 0.0, grads: dict | None = None, stream=None) -> dict:
        """Gradients of <dy, y> + L_aux + z_coef * z_loss after forward() on a
        config with save_for_backward (x must be unchanged since). Returns the
        fp32 gradient tensors (allocated on first use unless given)."""
        if grads is None:
            if getattr(self, "_grads", None) is None:
                self._grads = alloc_grads(self.cfg, self.b_r is not None, self.ws.device)
            grads = self._grads
        moe_backward(self.cfg, self._x, self.w_r, self.weights, dy, z_coef, grads, self.stats,
                     self.ws, stream)
        return grads

    def forward_host(self, x_host, y_host, x_dev, stream=None):
        """End-to-end call on host buffers: copy x (pinned host) in, run the
        layer, copy y and L_aux back; returns L_aux (a host float tensor)."""
        x_dev.copy_(x_host, non_blocking=True)
        self.forward(x_dev, stream)
        y_host.copy_(self.y, non_blocking=True)
        return self.stats.l_aux.to("cpu", non_blocking=True)

    def forward_host_stream(self, x_hosts, y_hosts, laux_host):
        """Runs the layer on a sequence of pinned host batches: y_hosts[i] =
        layer(x_hosts[i]) and laux_host[i] = its L_aux. The host-to-device copy
        of batch i+1 and the device-to-host copy of batch i-1 run on their own
        streams while batch i computes (two device buffers for x, y and the
        statistics). Returns when every copy has landed."""
        n = len(x_hosts)
        if n == 0:
            return
        dev = self.ws.device
        cfg = self.cfg
        if not hasattr(self, "_pipe"):
            mk = lambda: torch.empty((cfg.T, cfg.d_model), dtype=cfg.torch_dtype, device=dev)
            self._pipe = {"x": [mk(), mk()], "y": [mk(), mk()],
                          "stats": [Stats(cfg.n_experts, dev), Stats(cfg.n_experts, dev)],
                          "s_in": torch.cuda.Stream(dev), "s_out": torch.cuda.Stream(dev)}
        p = self._pipe
        comp = torch.cuda.current_stream(dev)
        in_done = [torch.cuda.Event(), torch.cuda.Event()]
        comp_done = [torch.cuda.Event(), torch.cuda.Event()]
        out_done = [torch.cuda.Event(), torch.cuda.Event()]
        for b in range(2):  # buffers start free
            comp_done[b].record(comp)
            out_done[b].record(comp)
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(p["s_in"]):
                p["s_in"].wait_event(comp_done[b])        # batch i-2 no longer reads x[b]
                p["x"][b].copy_(x_hosts[i], non_blocking=True)
                in_done[b].record(p["s_in"])
            comp.wait_event(in_done[b])
            comp.wait_event(out_done[b])                  # y[b] of batch i-2 copied out
            moe_forward(cfg, p["x"][b], self.w_r, self.b_r, self.weights, p["y"][b],
                        p["stats"][b], self.ws, comp)
            comp_done[b].record(comp)
            with torch.cuda.stream(p["s_out"]):
                p["s_out"].wait_event(comp_done[b])
                y_hosts[i].copy_(p["y"][b], non_blocking=True)
                laux_host[i:i + 1].copy_(p["stats"][b].l_aux, non_blocking=True)
                out_done[b].record(p["s_out"])
        p["s_out"].synchronize()


# --------------------------------------------------------------------------
# expert-parallel staging (the layout around the two all-to-alls; the caller
# exchanges the buffers with its own collective)
# --------------------------------------------------------------------------
def ep_workspace_size(cfg: LayerConfig, n_ranks: int) -> int:
    return int(load_library().moe_ep_workspace_size(ctypes.byref(cfg.c()), int(n_ranks)))


moe_ep_workspace_size = ep_workspace_size


def alloc_ep_workspace(cfg: LayerConfig, n_ranks: int, device="cuda") -> torch.Tensor:
    n = ep_workspace_size(cfg, n_ranks)
    if n == 0:
        raise MoEError(MOE_ERR_INVALID, "moe_ep_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _st(stats):
    return ctypes.byref(stats.c()) if stats is not None else None


def moe_ep_pack(cfg: LayerConfig, n_ranks: int, owner, offsets, x_perm, send, send_counts,
                stats: Stats | None, ws, stream=None):
    code = load_library().moe_ep_pack(ctypes.byref(cfg.c()), int(n_ranks), _ptr(owner),
                                      _ptr(offsets), _ptr(x_perm), _ptr(send),
                                      _ptr(send_counts), _st(stats), _ptr(ws), _stream(stream))
    _check(code, "moe_ep_pack")


def moe_ep_regroup(cfg: LayerConfig, n_ranks: int, rank: int, owner, kept_all, rows_cap: int,
                   recv, x_local, local_offsets, stats: Stats | None, ws, stream=None):
    code = load_library().moe_ep_regroup(ctypes.byref(cfg.c()), int(n_ranks), int(rank),
                                         _ptr(owner), _ptr(kept_all), int(rows_cap), _ptr(recv),
                                         _ptr(x_local), _ptr(local_offsets), _st(stats),
                                         _ptr(ws), _stream(stream))
    _check(code, "moe_ep_regroup")


def moe_ep_regroup_back(cfg: LayerConfig, n_ranks: int, rank: int, owner, kept_all,
                        rows_cap: int, o_local, back, stats: Stats | None, ws, stream=None):
    code = load_library().moe_ep_regroup_back(ctypes.byref(cfg.c()), int(n_ranks), int(rank),
                                              _ptr(owner), _ptr(kept_all), int(rows_cap),
                                              _ptr(o_local), _ptr(back), _st(stats), _ptr(ws),
                                              _stream(stream))
    _check(code, "moe_ep_regroup_back")


def moe_ep_unpack(cfg: LayerConfig, n_ranks: int, owner, offsets, back, o,
                  stats: Stats | None, ws, stream=None):
    code = load_library().moe_ep_unpack(ctypes.byref(cfg.c()), int(n_ranks), _ptr(owner),
                                        _ptr(offsets), _ptr(back), _ptr(o), _st(stats),
                                        _ptr(ws), _stream(stream))
    _check(code, "moe_ep_unpack")
