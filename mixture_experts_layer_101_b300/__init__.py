"""Sparse Mixture-of-Experts FFN layer (forward) for NVIDIA B300 (sm_103a).

The compute lives in libmoe.so (hand-written CUDA; C ABI in include/moe.h);
this package is its ctypes binding. Build the library with
`python -m mixture_experts_layer_101_b300.build`.
"""
from .moe import (EXPORTED, LIB_PATH, LayerConfig, MoEError, MoELayer, Stats, a_max, rows_max,
                  alloc_workspace, capacity, ffn_uses_tensor_cores, forward_launch_count, load_library, moe_combine,
                  moe_dispatch, moe_expert_ffn, moe_forward, moe_route, moe_route_no_workspace,
                  moe_status_string,
                  moe_trace_events, TRACE_STAGES, TraceEvents, moe_selftest_bounded_wait,
                  moe_workspace_size, status_string, workspace_size)

__all__ = ["EXPORTED", "LIB_PATH", "LayerConfig", "MoEError", "MoELayer", "Stats", "a_max", "rows_max",
           "alloc_workspace", "capacity", "ffn_uses_tensor_cores", "forward_launch_count", "load_library", "moe_combine",
           "moe_dispatch", "moe_expert_ffn", "moe_forward", "moe_route", "moe_route_no_workspace",
           "moe_status_string",
           "moe_trace_events", "TRACE_STAGES", "TraceEvents", "moe_selftest_bounded_wait",
           "moe_workspace_size", "status_string", "workspace_size"]
