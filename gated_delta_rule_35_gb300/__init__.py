"""GB300-native chunked forward of the gated delta rule (Gated DeltaNet).

    from gated_delta_rule_35_gb300 import chunk_fwd
    o, h_final = chunk_fwd(q, k, v, g, beta, scale, h0)

The compute runs in ``lib/libgdn.so`` (hand-written sm_103a kernels behind the
C ABI of ``include/gdn.h``); this package only marshals arguments.
"""
from .native import (GdnError, chunk_fwd, chunk_fwd_host, chunk_fwd_stages, check_device_status,
                     decode_step, problem, workspace_bytes)

__all__ = ["GdnError", "chunk_fwd", "chunk_fwd_host", "chunk_fwd_stages", "check_device_status",
           "decode_step", "problem", "workspace_bytes"]
