"""Beam routed-MoE forward pass for B300 (sm_103a).

The compute lives in libbeam_moe.so (hand-written CUDA; C ABI in include/beam_moe.h).
`abi` is its thin ctypes binding; `workloads` holds the seeded synthetic inputs;
`moe` offers a tensor-level convenience layer over the same calls.
"""
from . import workloads  # noqa: F401
from .abi import (  # noqa: F401
    BeamMoeConfig, BeamMoeError, beam_moe_default_config, beam_moe_dense_mlp, beam_moe_device_status,
    beam_moe_forward,
    beam_moe_forward_ex, beam_moe_forward_fp8, beam_moe_forward_shard, beam_moe_last_error, beam_moe_last_launch_count, beam_moe_route, beam_moe_route_ex,
    beam_moe_rmsnorm, beam_moe_route_noalloc, beam_moe_router_logits, beam_moe_sublayer_forward,
    beam_moe_timing_enable, beam_moe_timing_read,
)
