"""GB300-native Kimi Delta Attention (KDA) hot path: chunked prefill and pooled decode.

The compute path is libkda.so (hand-written CUDA for sm_103a, C-ABI in
include/kda.h); this package holds its in-tree build, a thin ctypes binding with
the same entry-point names, and the seeded synthetic-input generators.
"""
from .binding import (  # noqa: F401
    KdaError,
    kda_chunk_bwd,
    kda_chunk_fwd,
    kda_chunk_fwd_checkpoints,
    kda_chunk_fwd_workspace_size,
    kda_decode_multi,
    kda_decode_step,
    kda_get_device_error,
    kda_status_string,
    kda_trace_collect,
    kda_trace_enable,
    load_library,
)
