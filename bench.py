#!/usr/bin/env python
"""Benchmark of the sparse-MoE forward layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one moe_forward over one batch of the workload (router, capacity
dispatch, grouped expert FFN, combine, statistics) with every input resident
in HBM. The default workload is the Mixtral-shaped prefill layer (T=4096,
d=4096, N=8, K=2, SwiGLU F=14336, bf16), seeded synthetic data.

Timing: W untimed warm-up steps; then exactly K steps between a barrier and
a device synchronise on both sides. Before each step a 256 MB buffer is
written (L2 is 126 MB) outside the step's CUDA-event interval; the step time
is the interval between events recorded on the launch stream by the library
at the step's start and end. value = tokens of all ranks / max over ranks of
the summed step time. The library's trace events also time each stage; the
dominant kernel's roofline fraction uses that kernel's own interval. The
step (forward, or forward + backward with --pass train) is captured once as
a CUDA graph (the same kernels, the trace events recorded as graph nodes)
and replayed each step, with a synchronise after each replay, outside the
events, to read them; --eager launches every kernel per step instead.

e2e: the same metric through MoELayer.forward_host: pinned host x copied in,
the layer, y and L_aux copied out, per step, wall clock with a sync per step.

--impl reference: the float64 CPU oracle, unchanged, timed on this host's
cores on a bounded token sample of the same workload (rank 0 only).

--pass train: one step = moe_forward keeping its state + moe_backward (every
gradient of <dy, y> + L_aux + z_coef * z_loss) with a seeded dy; the metric
becomes training-step tokens/sec, and the roofline entry is the longest
kernel of the step.

With torchrun (N > 1) every rank runs its own replica of the layer on its
own GPU (the layer has no cross-token exchange): weak scaling, no collective
on the data path; only the timing is reduced across ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import moe_inputs  # noqa: E402

METRIC = "MoE-layer tokens/sec and % of roofline (TFLOP/s or HBM GB/s), 1×B300"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the dominant kernel, from an ncu capture of that kernel, valid only while
# the kernel sources hash to the fingerprint recorded with it (otherwise
# "traffic" is reported as null).
KERNEL_SOURCES = ["mixture_experts_layer_101_b300/csrc/ffn_tc.cu",
                  "mixture_experts_layer_101_b300/csrc/ptx_sm100.cuh",
                  "mixture_experts_layer_101_b300/csrc/moe_common.cuh"]
MEASURED_TRAFFIC = {("mixtral_prefill", "gate_up"): (1946806272 + 227520256, "b9c64ebbe0ff42d2"),
                    ("mixtral_prefill", "down"): (1429159680 + 122314752, "b9c64ebbe0ff42d2")}


def kernel_fingerprint() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]
UNIT = "tokens/s"
FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ----------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks during the timed region (read-only NVML queries)
# ----------------------------------------------------------------------------
class _NvmlReader:
    """Read-only NVML queries through ctypes (clock, max clock, clock-event
    reasons) for the GPU torch is using."""

    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        ok = False
        try:
            uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            ok = self.lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(),
                                                    ctypes.byref(self.handle)) == 0
        except Exception:
            ok = False
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.handle)) != 0:
            raise RuntimeError("no NVML device handle")
        try:
            self._reasons_fn = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self):
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, self.ct.byref(v))
        return int(v.value)

    def sm_max_mhz(self):
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.NVML_CLOCK_SM, self.ct.byref(v))
        return int(v.value)

    def reasons(self):
        v = self.ct.c_ulonglong()
        self._reasons_fn(self.handle, self.ct.byref(v))
        return int(v.value)


class ClockSampler:
    """Samples the SM clock and the clock-event reasons every few ms while the
    timed region runs (read-only; changes no GPU setting)."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock"}

    def __init__(self, period_s=0.005):
        self.period = period_s
        self.samples = []
        self.reason_bits = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self.error = None
        try:
            self.nvml = _NvmlReader()
            self.max_mhz = self.nvml.sm_max_mhz()
        except Exception as e:  # no NVML: report nothing rather than guess
            self.nvml = None
            self.error = f"nvml unavailable: {e}"

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nvml.sm_mhz())
                self.reason_bits |= self.nvml.reasons()
            except Exception as e:
                self.error = str(e)
                return
            time.sleep(self.period)

    def __enter__(self):
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()

    def summary(self):
        reasons = [name for bit, name in self.REASONS.items()
                   if self.reason_bits & bit and name != "gpu_idle"]
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
               "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples)}
        if self.error:
            out["note"] = self.error
        return out


# ----------------------------------------------------------------------------
# roofline bookkeeping
# ----------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained",
                                                     p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


def combine_fused(w) -> bool:
    """Whether moe_forward writes y from the down projection's epilogue: one
    expert output per token (K = 1, no shared experts) on the tensor-core path
    (bf16 SwiGLU, d % 256 == 0, F % 128 == 0)."""
    return (w.K == 1 and w.n_shared == 0 and w.dtype == "bf16" and w.activation == "swiglu"
            and w.d % 256 == 0 and w.F % 128 == 0)


def algorithmic_work(w, kept, offsets_active):
    """FLOPs and bytes the layer's definition needs (kept assignments only).

    gate/up GEMM: flops 2*A*d*(2F); bytes: the active experts' gate and up
    weights once, x_perm read once, h written once (bf16).
    down GEMM:    flops 2*A*F*d; bytes: active experts' down weights, h read,
                  o written (fp32); with the combine fused into it (K = 1, no
                  shared experts) y written for the kept tokens instead (and
                  their residual rows read).
    layer:        flops 2*A*d*F*mats; bytes: active experts' weights once, x
                  read once, y written once, the router weights."""
    A = int(kept)
    es = 2 if w.dtype == "bf16" else 4
    mats = 3 if w.activation == "swiglu" else 2
    act = int(offsets_active)
    d, F = w.d, w.F
    gu_flops = 2.0 * A * d * F * (2 if w.activation == "swiglu" else 1)
    gu_bytes = act * (mats - 1) * F * d * es + A * d * es + A * F * es
    dn_flops = 2.0 * A * F * d
    if combine_fused(w):
        dn_bytes = act * F * d * es + A * F * es + A * d * es * (2 if w.add_residual else 1)
    else:
        dn_bytes = act * F * d * es + A * F * es + A * d * 4
    layer_flops = gu_flops + dn_flops
    layer_bytes = act * mats * F * d * es + 2 * w.T * d * es + w.N * d * 4
    return {"gate_up": (gu_flops, gu_bytes), "down": (dn_flops, dn_bytes),
            "layer": (layer_flops, layer_bytes)}


def backward_work(w, kept, active):
    """FLOPs and bytes of the backward products (bf16 SwiGLU layers), per
    launch, and of the whole training step (forward + backward).
    down dgrad:    dh = dout W_down (2 A d F); reads the active down weights,
                   dout, the kept pre-activations, writes their gradients.
    down wgrad:    dW_down = dout^T h (2 A d F); reads dout, h; writes dW_down
                   of every expert (fp32).
    gate/up dgrad: dx_perm = da W_gate + db W_up (4 A d F); reads the active
                   gate and up weights and (da | db); writes dx_perm (fp32).
    gate/up wgrad: dW_gate, dW_up (4 A d F); reads (da | db), x_perm; writes
                   both gradients of every expert (fp32).
    step:          the forward's work, plus 2x its FLOPs; the weights read
                   again, every weight gradient written, dy read, dx written."""
    A, act = int(kept), int(active)
    d, F = w.d, w.F
    es = 2 if w.dtype == "bf16" else 4
    E = w.N + w.n_shared
    fwd = algorithmic_work(w, kept, active)
    out = {
        "bwd_down_dgrad": (2.0 * A * d * F, act * F * d * es + A * d * es + 2 * A * 2 * F * es),
        "bwd_down_wgrad": (2.0 * A * d * F, A * d * es + A * F * es + E * d * F * 4),
        "bwd_gate_up_dgrad": (4.0 * A * d * F, 2 * act * F * d * es + A * 2 * F * es + A * d * 4),
        "bwd_gate_up_wgrad": (4.0 * A * d * F, A * 2 * F * es + A * d * es + E * 2 * F * d * 4),
    }
    fl, by = fwd["layer"]
    out["step"] = (3.0 * fl, by + act * 3 * F * d * es + E * 3 * F * d * 4 +
                   w.T * d * (es + 4) + 2 * w.N * d * 4)
    return out


def roofline_entry(flops, nbytes, seconds, peaks, sustained=False):
    """The bound (tensor or HBM) whose roofline time is larger, with the
    achieved rate and its fraction of the measured peak. sustained selects the
    measured power-capped bf16 rate instead of the burst rate."""
    tflops_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    t_tensor = flops / (tflops_peak * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        ach = flops / seconds / 1e12
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": tflops_peak,
                "unit": "TFLOP/s", "frac": round(ach / tflops_peak, 4)}
    ach = nbytes / seconds / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4)}


# ----------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ----------------------------------------------------------------------------
F64_HOST_LIMIT = 16 << 30


def host_inputs(w, experts_dev=None):
    """The workload's inputs on the host. Expert weights are handed to the
    oracle already in float64 when that fits in F64_HOST_LIMIT bytes (the
    oracle's own promotion is then a no-op); otherwise the oracle promotes
    each expert it needs, inside the timed call."""
    x = moe_inputs.make_x(w)
    w_r, b_r = moe_inputs.make_router(w)
    if experts_dev is not None:
        experts = {k: v.cpu() for k, v in experts_dev.items()}
    elif torch.cuda.is_available():
        experts = {k: v.cpu() for k, v in moe_inputs.make_experts(w, "cuda").items()}
    else:
        experts = moe_inputs.make_experts(w, "cpu")
    if sum(v.numel() for v in experts.values()) * 8 <= F64_HOST_LIMIT:
        experts = {k: v.double().numpy() for k, v in experts.items()}
    return x, w_r, b_r, experts


def time_oracle(w, x, w_r, b_r, experts, n_tokens):
    """One call of the oracle as it stands: routing, statistics and dispatch
    of every token, expert FFN and combine of the first n_tokens tokens."""
    from oracle import moe_oracle as O
    t0 = time.perf_counter()
    O.moe_forward(x, w_r, b_r, lambda e: {k: v[e] for k, v in experts.items()}, K=w.K,
                  activation=w.activation, capacity_factor=w.capacity_factor, alpha=w.alpha,
                  add_residual=w.add_residual, tokens=range(n_tokens), gate_mode=w.gate_mode,
                  select_bias=moe_inputs.make_select_bias(w))
    return time.perf_counter() - t0


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, experts_dev, budget_s=15.0):
    x, w_r, b_r, experts = host_inputs(w, experts_dev)
    n = min(w.T, 64)
    t = time_oracle(w, x, w_r, b_r, experts, n)
    # grow the sample towards the time budget (bounded by the workload)
    while n < w.T and t < budget_s / 4:
        n = min(w.T, n * 4)
        t = time_oracle(w, x, w_r, b_r, experts, n)
    pre = isinstance(next(iter(experts.values())), __import__("numpy").ndarray)
    return {"value": round(n / t, 3), "unit": UNIT, "cores": cores_used(), "kind": "oracle",
            "sample": f"float64 oracle: routing/statistics/dispatch of all {w.T} tokens, "
                      f"experts and combine of the first {n} tokens; {t:.2f} s; "
                      f"value = {n} tokens / that time; expert weights "
                      + ("given in float64" if pre else "promoted by the oracle per call")}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = selected_workload(args)
    x, w_r, b_r, experts = host_inputs(w)
    n = min(w.T, args.ref_tokens)
    for _ in range(args.warmup):
        time_oracle(w, x, w_r, b_r, experts, n)
    times = [time_oracle(w, x, w_r, b_r, experts, n) for _ in range(args.steps)]
    total = sum(times)
    value = n * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args, extra={"reference_sample_tokens": n}),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores_used(),
                             "kind": "oracle",
                             "sample": f"each step: routing of all {w.T} tokens and experts"
                                       f" + combine of the first {n} tokens, float64"},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, args, extra=None):
    cfg = {"workload": w.name, "T": w.T, "d_model": w.d, "d_ff": w.F, "n_experts": w.N,
           "top_k": w.K, "activation": w.activation, "capacity_factor":
           (None if math.isinf(w.capacity_factor) else w.capacity_factor),
           "residual": w.add_residual, "gate_mode": w.gate_mode,
           "select_bias": w.select_bias != "none", "parallelism": f"replicas x{args.gpus}",
           "l2": "256 MB written before every step, outside the step's event interval; "
                 "expert weights exceed L2"}
    if extra:
        cfg.update(extra)
    return cfg


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def selected_workload(args):
    import dataclasses
    w = moe_inputs.WORKLOADS[args.workload]
    w = dataclasses.replace(w, gate_mode=args.gate_mode,
                            select_bias="uniform" if args.select_bias else "none")
    if args.tokens is not None:  # a smaller batch of the same layer (profiling captures)
        w = dataclasses.replace(w, T=args.tokens)
    if args.experts is not None:  # fewer experts of the same shape (profiling captures)
        w = dataclasses.replace(w, N=args.experts, K=min(w.K, args.experts))
    return w


def run_ours(args, world, rank):
    import mixture_experts_layer_101_b300 as moe

    moe.load_library()
    w = selected_workload(args)
    cfg = moe.LayerConfig.from_workload(w)
    dev = torch.device("cuda", torch.cuda.current_device())
    sb = moe_inputs.make_select_bias(w)
    cfg.select_bias = None if sb is None else sb.to(dev)
    x = moe_inputs.make_x(w).to(dev)
    w_r, b_r = moe_inputs.make_router(w)
    w_r = w_r.to(dev)
    b_r = None if b_r is None else b_r.to(dev)
    experts = moe_inputs.make_experts(w, dev)
    layer = moe.MoELayer(cfg, w_r, b_r, experts, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    nst = len(moe.TRACE_STAGES) + 1
    for _ in range(args.warmup):
        layer.forward(x)
    torch.cuda.synchronize()
    layer.stats.status.zero_()

    if args.graph:
        # the step as one CUDA graph (captured with one set of stage events,
        # re-recorded by every replay and read after it)
        ev = moe.TraceEvents(nst)
        moe.moe_trace_events(ev.handles())
        graph = layer.capture(x)
        moe.moe_trace_events([])
        torch.cuda.synchronize()
        layer.stats.status.zero_()
    else:
        events = [moe.TraceEvents(nst) for _ in range(args.steps)]
    step_ms, stage_ms = [], {name: [] for name in moe.TRACE_STAGES}
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler() as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            if args.graph:
                graph.replay()
                torch.cuda.synchronize()  # outside the events: the replay's own times
                step_ms.append(ev.elapsed_ms(0, nst - 1))
                for j, name in enumerate(moe.TRACE_STAGES):
                    stage_ms[name].append(ev.elapsed_ms(j, j + 1))
            else:
                moe.moe_trace_events(events[i].handles())
                layer.forward(x)
        moe.moe_trace_events([])
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(world)

    if not args.graph:
        step_ms = [ev.elapsed_ms(0, nst - 1) for ev in events]
        stage_ms = {name: [ev.elapsed_ms(j, j + 1) for ev in events]
                    for j, name in enumerate(moe.TRACE_STAGES)}
    dev_s = sum(step_ms) / 1e3
    max_s = max_over_ranks(dev_s, world)
    tokens = sum_over_ranks(float(w.T * args.steps), world)
    value = tokens / max_s

    st = layer.stats.to_host()
    if st["status"] != 0:
        raise SystemExit(f"device status word {st['status']:#x} after the timed steps")
    # shared experts process every token: T more rows each, always active
    kept = int(st["kept"].sum()) + w.n_shared * w.T
    active = int((st["kept"] > 0).sum()) + w.n_shared
    work = algorithmic_work(w, kept, active)
    peaks = measured_peaks()
    gu_s = statistics.mean(stage_ms["ffn_gate_up"]) / 1e3
    dn_s = statistics.mean(stage_ms["ffn_down"]) / 1e3
    dominant = "ffn_gate_up" if gu_s >= dn_s else "ffn_down"
    key = "gate_up" if dominant == "ffn_gate_up" else "down"
    # A run that the power cap held well below the maximum SM clock is a
    # sustained run: its tensor roofline is the measured sustained bf16 rate.
    ck = clocks.summary()
    sustained = ("sw_power_cap" in ck["reasons"] and ck["sm_mhz"] is not None and
                 ck["sm_max_mhz"] and ck["sm_mhz"] < 0.9 * ck["sm_max_mhz"])
    kern_s = gu_s if key == "gate_up" else dn_s
    roof = roofline_entry(*work[key], kern_s, peaks, sustained)
    roof["kernel"] = ("grouped expert GEMM gate/up + SwiGLU" if key == "gate_up"
                      else "grouped expert GEMM down")
    meas = MEASURED_TRAFFIC.get((w.name, key))
    roof["traffic"] = (meas[0] if meas is not None and meas[1] == kernel_fingerprint()
                       else None)
    roof["peak_source"] = (f"{peaks['source']} bf16 "
                           + ("sustained (run power-capped)" if sustained else "burst")
                           if roof["bound"] == "tensor" else f"{peaks['source']} HBM copy")
    if roof["bound"] == "tensor":
        roof["frac_of_burst_peak"] = round(work[key][0] / kern_s / 1e12 / peaks["bf16_tflops"], 4)
    layer_roof = roofline_entry(*work["layer"], statistics.mean(step_ms) / 1e3, peaks, sustained)

    # end to end through the public API on host buffers: every step copies
    # its batch in from pinned host memory and its y and L_aux out; copies of
    # neighbouring steps overlap the compute (MoELayer.forward_host_stream)
    e2e_steps = args.steps
    x_host = moe_inputs.make_x(w).pin_memory()
    x_hosts = [x_host] * e2e_steps
    y_hosts = [torch.empty((w.T, w.d), dtype=cfg.torch_dtype).pin_memory() for _ in range(2)]
    y_hosts = [y_hosts[i & 1] for i in range(e2e_steps)]
    laux_host = torch.empty(e2e_steps, dtype=torch.float32).pin_memory()
    layer.forward_host_stream(x_hosts[:min(args.warmup, 3)], y_hosts, laux_host)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    layer.forward_host_stream(x_hosts, y_hosts, laux_host)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier(world)
    if not bool(torch.isfinite(laux_host).all()):
        raise SystemExit("non-finite L_aux in the end-to-end run")
    e2e_value = sum_over_ranks(float(w.T * e2e_steps), world) / max_over_ranks(e2e_s, world)
    es = 2 if w.dtype == "bf16" else 4

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, experts)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * max_s / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": workload_config(w, args, {"launch": "cuda_graph" if args.graph else
                                                  "stream"}),
            "roofline": roof,
            "layer_roofline": dict(layer_roof, note="whole step against max(F/peak, B/BW) "
                                                    "of the layer's algorithmic work"),
            "stage_ms": {k: round(statistics.mean(v), 4) for k, v in stage_ms.items()},
            "kept_assignments": kept, "active_experts": active, "n_dropped": st["n_dropped"],
            "l_aux": st["l_aux"],
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT,
                    "h2d_bytes_per_step": w.T * w.d * es,
                    "d2h_bytes_per_step": w.T * w.d * es + 4},
            "gpu_launches": moe.forward_launch_count(cfg) * args.steps,
            "clocks": ck,
            "wall_s_timed_region": round(wall, 4),
        }
        print(json.dumps(line), flush=True)
    return 0


def run_train(args, world, rank):
    """Training step: moe_forward (keeping its state) + moe_backward."""
    import mixture_experts_layer_101_b300 as moe

    moe.load_library()
    w = selected_workload(args)
    if w.dtype != "bf16" or w.activation != "swiglu":
        raise SystemExit("--pass train times bf16 SwiGLU layers")
    cfg = moe.LayerConfig.from_workload(w)
    cfg.save_for_backward = True
    dev = torch.device("cuda", torch.cuda.current_device())
    sb = moe_inputs.make_select_bias(w)
    cfg.select_bias = None if sb is None else sb.to(dev)
    x = moe_inputs.make_x(w).to(dev)
    dy = moe_inputs.make_dy(w).to(dev)
    w_r, b_r = moe_inputs.make_router(w)
    w_r = w_r.to(dev)
    b_r = None if b_r is None else b_r.to(dev)
    experts = moe_inputs.make_experts(w, dev)
    layer = moe.MoELayer(cfg, w_r, b_r, experts, device=dev)
    grads = moe.alloc_grads(cfg, b_r is not None, dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    z = args.z_coef
    nf, nb = len(moe.TRACE_STAGES) + 1, len(moe.TRACE_STAGES_BWD) + 1

    for _ in range(args.warmup):
        layer.forward(x)
        layer.backward(dy, z, grads)
    torch.cuda.synchronize()

    def step(h):
        moe.moe_trace_events(h[:nf])
        layer.forward(x)
        moe.moe_trace_events(h[nf:])
        layer.backward(dy, z, grads)
        moe.moe_trace_events([])

    def times(ev):
        out = {name: ev.elapsed_ms(j, j + 1) for j, name in enumerate(moe.TRACE_STAGES)}
        out.update({name: ev.elapsed_ms(nf + j, nf + j + 1)
                    for j, name in enumerate(moe.TRACE_STAGES_BWD)})
        return ev.elapsed_ms(0, nf + nb - 1), out

    if args.graph:  # forward + backward captured once, replayed per step
        ev = moe.TraceEvents(nf + nb)
        graph = moe.capture_graph(lambda: step(ev.handles()), dev)
    else:
        events = [moe.TraceEvents(nf + nb) for _ in range(args.steps)]
    torch.cuda.synchronize()
    layer.stats.status.zero_()
    step_ms, stage_ms = [], {n: [] for n in (*moe.TRACE_STAGES, *moe.TRACE_STAGES_BWD)}
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler() as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            if args.graph:
                graph.replay()
                torch.cuda.synchronize()  # outside the events: the replay's own times
                t, st_i = times(ev)
                step_ms.append(t)
                for k, v in st_i.items():
                    stage_ms[k].append(v)
            else:
                step(events[i].handles())
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(world)
    if not args.graph:
        for e in events:
            t, st_i = times(e)
            step_ms.append(t)
            for k, v in st_i.items():
                stage_ms[k].append(v)
    max_s = max_over_ranks(sum(step_ms) / 1e3, world)
    value = sum_over_ranks(float(w.T * args.steps), world) / max_s
    st = layer.stats.to_host()
    if st["status"] != 0:
        raise SystemExit(f"device status word {st['status']:#x} after the timed steps")
    if not all(bool(torch.isfinite(g).all()) for g in grads.values() if g is not None):
        raise SystemExit("non-finite gradient after the timed steps")
    kept = int(st["kept"].sum()) + w.n_shared * w.T
    active = int((st["kept"] > 0).sum()) + w.n_shared
    fw, bw = algorithmic_work(w, kept, active), backward_work(w, kept, active)
    work = {"ffn_gate_up": fw["gate_up"], "ffn_down": fw["down"], **bw}
    means = {k: statistics.mean(v) / 1e3 for k, v in stage_ms.items()}
    dominant = max((k for k in work if k in means), key=lambda k: means[k])
    ck = clocks.summary()
    sustained = ("sw_power_cap" in ck["reasons"] and ck["sm_mhz"] is not None and
                 ck["sm_max_mhz"] and ck["sm_mhz"] < 0.9 * ck["sm_max_mhz"])
    peaks = measured_peaks()
    roof = roofline_entry(*work[dominant], means[dominant], peaks, sustained)
    roof["kernel"] = dominant
    roof["traffic"] = None
    roof["peak_source"] = (f"{peaks['source']} bf16 "
                           + ("sustained (run power-capped)" if sustained else "burst")
                           if roof["bound"] == "tensor" else f"{peaks['source']} HBM copy")
    step_roof = roofline_entry(*bw["step"], statistics.mean(step_ms) / 1e3, peaks, sustained)

    # end to end on host buffers: x and dy copied in from pinned memory, dx
    # and L_aux copied out, every step
    es = 2
    x_h = moe_inputs.make_x(w).pin_memory()
    dy_h = moe_inputs.make_dy(w).pin_memory()
    dx_h = torch.empty((w.T, w.d), dtype=torch.float32).pin_memory()
    laux_h = torch.empty(1, dtype=torch.float32).pin_memory()
    x_d, dy_d = torch.empty_like(x), torch.empty_like(dy)

    def e2e_step():
        x_d.copy_(x_h, non_blocking=True)
        dy_d.copy_(dy_h, non_blocking=True)
        layer.forward(x_d)
        layer.backward(dy_d, z, grads)
        dx_h.copy_(grads["dx"], non_blocking=True)
        laux_h.copy_(layer.stats.l_aux, non_blocking=True)

    for _ in range(min(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier(world)
    e2e_value = sum_over_ranks(float(w.T * args.steps), world) / max_over_ranks(e2e_s, world)

    if rank == 0:
        line = {
            "metric": "MoE-layer training-step tokens/sec (forward + backward) and % of "
                      "roofline, 1×B300",
            "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * max_s / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": workload_config(w, args, {"pass": "train", "z_coef": z,
                                                  "launch": "cuda_graph" if args.graph else
                                                  "stream"}),
            "roofline": roof,
            "step_roofline": dict(step_roof, note="whole training step against "
                                                  "max(F/peak, B/BW) of its algorithmic work"),
            "stage_ms": {k: round(statistics.mean(v), 4) for k, v in stage_ms.items()},
            "kept_assignments": kept, "active_experts": active,
            "cpu_baseline": None,
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT,
                    "h2d_bytes_per_step": 2 * w.T * w.d * es,
                    "d2h_bytes_per_step": w.T * w.d * 4 + 4},
            # moe_backward_launch_count counts the router-bias gradient (2 kernels)
            "gpu_launches": (moe.forward_launch_count(cfg) + moe.backward_launch_count(cfg)
                             - (0 if b_r is not None else 2)) * args.steps,
            "clocks": ck,
            "wall_s_timed_region": round(wall, 4),
        }
        print(json.dumps(line), flush=True)
    return 0


def ep_bytes(rows_src, rows_dst, d, es):
    """Bytes each expert-parallel staging call reads plus writes: pack and
    unpack move the source device's kept rows (x in the layer dtype, expert
    outputs in fp32), regroup and regroup back the rows a device receives."""
    return {"ep_pack": 2 * rows_src * d * es, "ep_unpack": 2 * rows_src * d * 4,
            "ep_regroup": 2 * rows_dst * d * es, "ep_regroup_back": 2 * rows_dst * d * 4}


def run_ep(args, world, rank):
    """Expert-parallel staging on one device: the source side (pack of the
    dispatched rows by destination, unpack of the returned fp32 outputs) and
    the destination side of device 0 (regroup of what it receives by expert,
    regroup back of its outputs), with args.ep_ranks devices holding the
    experts in blocks and every source routing like this one. The exchange
    itself is not part of the library and not timed."""
    import mixture_experts_layer_101_b300 as moe

    moe.load_library()
    w = selected_workload(args)
    if w.n_shared:
        raise SystemExit("--pass ep: shared experts are not exchanged")
    R = args.ep_ranks
    cfg = moe.LayerConfig.from_workload(w)
    dev = torch.device("cuda", torch.cuda.current_device())
    x = moe_inputs.make_x(w).to(dev)
    w_r, b_r = moe_inputs.make_router(w)
    N, K, d = w.N, w.K, w.d
    ws = moe.alloc_workspace(cfg, dev)
    st = moe.Stats(N, dev)
    A = max(moe.a_max(cfg), 1)
    idx = torch.empty((w.T, K), dtype=torch.int32, device=dev)
    gate = torch.empty((w.T, K), dtype=torch.float32, device=dev)
    moe.moe_route(cfg, x, w_r.to(dev), None if b_r is None else b_r.to(dev), idx, gate, st, ws)
    offsets = torch.empty(N + 1, dtype=torch.int32, device=dev)
    slot_of = torch.empty((w.T, K), dtype=torch.int32, device=dev)
    tos = torch.empty(A, dtype=torch.int32, device=dev)
    x_perm = torch.empty((A, d), dtype=cfg.torch_dtype, device=dev)
    moe.moe_dispatch(cfg, x, idx, offsets, slot_of, tos, x_perm, st, ws)
    torch.cuda.synchronize()
    owner_h = [e * R // N for e in range(N)]
    owner = torch.tensor(owner_h, dtype=torch.int32, device=dev)
    kept = st.kept.clone()
    kept_all = kept.unsqueeze(0).repeat(R, 1).contiguous()
    rows_src = int(kept.sum())
    rows_dst = R * int(sum(int(kept[e]) for e in range(N) if owner_h[e] == 0))
    cap = max(rows_dst, 1)
    g = torch.Generator(device=dev).manual_seed(7)
    send = torch.empty((A, d), dtype=cfg.torch_dtype, device=dev)
    counts = torch.empty(R, dtype=torch.int32, device=dev)
    back = torch.randn((A, d), generator=g, device=dev)
    o = torch.empty((A, d), dtype=torch.float32, device=dev)
    recv = torch.randn((cap, d), generator=g, device=dev).to(cfg.torch_dtype)
    x_local = torch.empty((cap, d), dtype=cfg.torch_dtype, device=dev)
    loff = torch.empty(N + 1, dtype=torch.int32, device=dev)
    o_local = torch.randn((cap, d), generator=g, device=dev)
    back_local = torch.empty((cap, d), dtype=torch.float32, device=dev)
    ws_ep = moe.alloc_ep_workspace(cfg, R, dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    calls = {
        "ep_pack": lambda: moe.moe_ep_pack(cfg, R, owner, offsets, x_perm, send, counts, st,
                                           ws_ep),
        "ep_regroup": lambda: moe.moe_ep_regroup(cfg, R, 0, owner, kept_all, cap, recv, x_local,
                                                 loff, st, ws_ep),
        "ep_regroup_back": lambda: moe.moe_ep_regroup_back(cfg, R, 0, owner, kept_all, cap,
                                                           o_local, back_local, st, ws_ep),
        "ep_unpack": lambda: moe.moe_ep_unpack(cfg, R, owner, offsets, back, o, st, ws_ep),
    }
    for _ in range(args.warmup):
        for f in calls.values():
            f()
    torch.cuda.synchronize()
    st.status.zero_()
    names = list(calls)
    ms = {n: [] for n in names}
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler() as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
            flush.fill_(i & 0xFF)
            ev[0].record()
            for j, n in enumerate(names):
                calls[n]()
                ev[j + 1].record()
            torch.cuda.synchronize()
            for j, n in enumerate(names):
                ms[n].append(ev[j].elapsed_time(ev[j + 1]))
        wall = time.perf_counter() - wall0
    barrier(world)
    if st.status_bits() != 0:
        raise SystemExit(f"device status word {st.status_bits():#x} after the timed steps")
    es = 2 if w.dtype == "bf16" else 4
    nbytes = ep_bytes(rows_src, rows_dst, d, es)
    mean_s = {n: statistics.mean(v) / 1e3 for n, v in ms.items()}
    step_s = sum(mean_s.values())
    max_s = max_over_ranks(step_s * args.steps, world)
    rows = 2 * rows_src + 2 * rows_dst
    value = sum_over_ranks(float(rows * args.steps), world) / max_s
    peaks = measured_peaks()
    dominant = max(names, key=lambda n: mean_s[n])
    roof = roofline_entry(0.0, nbytes[dominant], mean_s[dominant], peaks)
    roof.update(kernel=dominant, traffic=None, peak_source=f"{peaks['source']} HBM copy")
    per_call = {n: {"ms": round(mean_s[n] * 1e3, 4), "bytes": nbytes[n],
                    "gbs": round(nbytes[n] / mean_s[n] / 1e9, 1),
                    "frac": round(nbytes[n] / mean_s[n] / 1e9 / peaks["hbm_gbs"], 4)}
                for n in names}
    if rank == 0:
        line = {"metric": "EP staging rows/s (pack, regroup, regroup back, unpack), 1xB300",
                "value": round(value, 1), "unit": "rows/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
                "config": workload_config(w, args, {"ep_ranks": R, "placement": "block",
                                                    "source_rows": rows_src,
                                                    "received_rows": rows_dst}),
                "roofline": roof, "calls": per_call, "gpu_launches": 8 * args.steps,
                "clocks": clocks.summary(), "wall_s_timed_region": round(wall, 4)}
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="mixtral_prefill", choices=sorted(moe_inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=256,
                    help="tokens whose experts the reference arm evaluates per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gate-mode", default="renorm", choices=["renorm", "softmax"],
                    help="renorm: softmax over the K selected logits; softmax: full-softmax gate")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (small profiling cases)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override the workload's expert count (small profiling cases)")
    ap.add_argument("--eager", dest="graph", action="store_false",
                    help="launch every kernel per step instead of replaying the step as one "
                         "captured CUDA graph (the default)")
    ap.add_argument("--pass", dest="pass_", default="forward",
                    choices=["forward", "train", "ep"],
                    help="forward (the layer's metric), train: forward + backward, or ep: the "
                         "expert-parallel staging calls")
    ap.add_argument("--ep-ranks", type=int, default=8,
                    help="devices holding the experts (--pass ep)")
    ap.add_argument("--z-coef", type=float, default=1e-3,
                    help="z-loss weight in the training objective (--pass train)")
    ap.add_argument("--select-bias", action="store_true",
                    help="add a seeded top-K selection bias (auxiliary-loss-free balancing)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("at least 3 warm-up steps")
    world, rank, _ = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        if args.pass_ == "train":
            return run_train(args, world, rank)
        if args.pass_ == "ep":
            return run_ep(args, world, rank)
        return run_ours(args, world, rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
