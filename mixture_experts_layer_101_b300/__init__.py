"""Sparse Mixture-of-Experts FFN layer (forward and backward) for NVIDIA B300
(sm_103a).

The compute lives in libmoe.so (hand-written CUDA; C ABI in include/moe.h);
this package is its ctypes binding. Build the library with
`python -m mixture_experts_layer_101_b300.build`.
"""
from .moe import (EXPORTED, GRAD_NAMES, LIB_PATH, TRACE_STAGES, TRACE_STAGES_BWD, LayerConfig,
                  MoEError, MoELayer, Stats, TraceEvents, a_max, alloc_ep_workspace, alloc_grads,
                  alloc_workspace, ep_workspace_size, moe_ep_pack, moe_ep_regroup,
                  moe_ep_regroup_back, moe_ep_unpack, moe_ep_workspace_size,
                  backward_launch_count, capacity, capture_graph, ffn_uses_tensor_cores,
                  forward_launch_count, load_library, moe_backward, moe_backward_launch_count,
                  moe_combine, moe_dispatch, moe_expert_ffn, moe_forward, moe_route,
                  moe_route_no_workspace, moe_selftest_bounded_wait, moe_status_string,
                  moe_trace_events, moe_workspace_size, rows_max, status_string, workspace_size)

__all__ = ["EXPORTED", "GRAD_NAMES", "LIB_PATH", "TRACE_STAGES", "TRACE_STAGES_BWD",
           "LayerConfig", "MoEError", "MoELayer", "Stats", "TraceEvents", "a_max",
           "alloc_ep_workspace", "alloc_grads", "ep_workspace_size", "moe_ep_pack",
           "moe_ep_regroup", "moe_ep_regroup_back", "moe_ep_unpack", "moe_ep_workspace_size",
           "alloc_workspace", "backward_launch_count", "capacity", "capture_graph",
           "ffn_uses_tensor_cores", "forward_launch_count", "load_library", "moe_backward",
           "moe_backward_launch_count", "moe_combine", "moe_dispatch", "moe_expert_ffn",
           "moe_forward", "moe_route", "moe_route_no_workspace", "moe_selftest_bounded_wait",
           "moe_status_string", "moe_trace_events", "moe_workspace_size", "rows_max",
           "status_string", "workspace_size"]
