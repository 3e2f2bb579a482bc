"""fp64 input front-end of the oracle: the two steps that the problem flags
GDN_FLAG_RAW_G and GDN_FLAG_QK_L2NORM move into the kernels.

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline); it shares no code
with the CUDA path.

  chunk_cumsum   per-token log decays gamma -> the chunk-local cumulative sum
                 g the chunked form consumes: within each chunk of C tokens,
                 g_t is the sum of gamma over the chunk's tokens up to and
                 including t (the workloads' g is built the same way).
  l2norm_rows    each row x (the K values of one token of one head) becomes
                 x / sqrt(sum_i x_i^2 + eps), eps = 1e-6: the q/k
                 normalisation of the "KdaSplit" decode kernel page (its
                 per-token factors rsqrt(sum + 1e-6)); there, scale multiplies
                 the normalised q, which is what the forward's scale
                 argument does to o.
  prepare        both, as the flags select, ahead of ``recurrence.forward``
                 or ``chunked.forward``.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def chunk_cumsum(gamma, chunk: int = 64) -> np.ndarray:
    """[B, T, ...] per-token log decays -> chunk-local inclusive sums over T."""
    gamma = np.asarray(gamma, dtype=np.float64)
    g = np.empty_like(gamma)
    for s in range(0, gamma.shape[1], chunk):
        g[:, s:s + chunk] = np.cumsum(gamma[:, s:s + chunk], axis=1)
    return g


def l2norm_rows(x, eps: float = EPS) -> np.ndarray:
    """Rows over the last axis divided by sqrt(sum of squares + eps)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def prepare(q, k, g, *, raw_g: bool, qk_l2norm: bool, chunk: int = 64):
    """(q, k, g) as the forward consumes them, in fp64."""
    q, k, g = (np.asarray(a, dtype=np.float64) for a in (q, k, g))
    if qk_l2norm:
        q, k = l2norm_rows(q), l2norm_rows(k)
    if raw_g:
        g = chunk_cumsum(g, chunk)
    return q, k, g
