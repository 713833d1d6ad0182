"""GB300-native (sm_103a) Mixture-of-Experts layer forward.

route -> routing metadata -> grouped SwiGLU / SwiGLU-OAI / ReLU2 expert FFN
-> gate-weighted combine, every stage a CUDA kernel in libmoe_gb300.so
behind the C ABI of include/moe.h. This package is the thin Python binding
(argument marshalling over torch tensors) and nothing else; the seeded
synthetic inputs that tests and the benchmark use live in the top-level
`moe_inputs` module, outside the product.
"""
from ._binding import (ACT, FFN_KERNEL, GATING, LAYOUT, MoEError, MoeParams, RoutingMeta,
                       STAGES, build_metadata, combine, empty_meta, forward, forward_gate,
                       ffn_plan, forward_launch_count, forward_timed, grouped_ffn, lib, library_path,
                       make_params, read_status, route, route_gemm, route_metadata,
                       selftest_wait_timeout, status_string, workspace, workspace_regions,
                       workspace_size)

__all__ = ["ACT", "FFN_KERNEL", "GATING", "LAYOUT", "MoEError", "MoeParams", "RoutingMeta",
           "STAGES", "build_metadata", "combine", "empty_meta", "forward", "forward_gate",
           "ffn_plan", "forward_launch_count", "forward_timed", "grouped_ffn", "lib", "library_path",
           "make_params", "read_status", "route", "route_gemm", "route_metadata",
           "selftest_wait_timeout", "status_string", "workspace", "workspace_regions",
           "workspace_size"]
