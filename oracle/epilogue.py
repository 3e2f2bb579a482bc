"""fp64 gated RMSNorm of the output, the step after chunk_fwd_o in a Gated
DeltaNet layer.

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline); it shares no code
with the CUDA path.

Each output row o (the V values of one token of one head) becomes

    o * rstd * weight * sigmoid(gate),   rstd = 1 / sqrt(mean_v o_v^2 + eps)

as in the output stage of the "KdaSplit" decode kernel page (its root of the
mean square over the head's channels plus eps, times the norm weight and the
token's gate after a sigmoid). The logistic function comes from scipy.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit


def gated_rmsnorm(o, gate, weight, eps: float) -> np.ndarray:
    """o, gate [..., V]; weight [V]; returns the normalised, gated rows (fp64)."""
    o = np.asarray(o, dtype=np.float64)
    gate = np.asarray(gate, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    rstd = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o * rstd * weight * expit(gate)
