"""Seeded synthetic inputs for the CSA2 hot path.

This module only draws random numbers and names workload shapes. It holds
none of the method's arithmetic (no quantisation rule, no scoring, no
selection, no attention). Both the CUDA library's tests/benchmark and the
CPU oracle take their inputs from here.

Every tensor is drawn from its own ``torch.Generator`` seeded with
``seed * 1_000_003 + stream_id`` so that a tensor can be regenerated alone.
Values drawn on a CUDA device differ from values drawn on the CPU for the
same seed; callers that need both sides to see the same bytes draw once and
copy.
"""
from .gen import (
    STREAMS,
    gen_for,
    normal_bf16,
    uniform_f32,
    normal_e4m3,
    indexer_keys_e4m3,
)
from .configs import CONFIGS, Config, get_config

__all__ = [
    "STREAMS", "gen_for", "normal_bf16", "uniform_f32", "normal_e4m3",
    "indexer_keys_e4m3", "CONFIGS", "Config", "get_config",
]
