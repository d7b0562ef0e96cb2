"""GB300-native Gated DeltaNet (GDN) causal core.

The compute lives in libgdn.so (hand-written CUDA for sm_103a, C ABI in
include/gdn.h); this package is its torch-facing binding:

    from gated_deltanet_layer_causal_gb300 import gdn_core
    y, final_state = gdn_core(x, conv_w, a, b, A_log, dt_bias, z, norm_w,
                              cu_seqlens, h_k, h_v, output_final_state=True)

Lower-level entry points mirror the C ABI: conv1d_silu(_bwd), chunk_fwd,
chunk_bwd, gated_rmsnorm(_bwd), recurrent_step.  GDNLayer wraps the core in
its input and output projections (the whole layer).
"""
from .core import (GDNCore, chunk_bwd, chunk_fwd, conv1d_silu, conv1d_silu_bwd, gated_rmsnorm,
                   gated_rmsnorm_bwd, gdn_core, read_status, recurrent_step, workspace_size)
from .layer import GDNLayer

__all__ = ["GDNCore", "GDNLayer", "gdn_core", "conv1d_silu", "conv1d_silu_bwd", "chunk_fwd", "chunk_bwd",
           "gated_rmsnorm", "gated_rmsnorm_bwd", "recurrent_step", "read_status",
           "workspace_size"]
