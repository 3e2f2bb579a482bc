"""fp64 NumPy chunked form of the gated delta rule forward.

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline); it shares no code
with the CUDA path.

It follows the pipeline of the "WarpDrive" page (kernels 3-5, section
"Pipeline": recompute_w_u -> chunk_fwd_h -> chunk_fwd_o, chunk size C=64), one
chunk at a time, in the pages' notation, and exports every intermediate so
the CUDA stages can be compared one by one:

  A      per chunk, A = (I + L)^-1 with L the strictly lower gated Gram matrix
         L_ij = beta_i (k_i . k_j) exp(g_i - g_j) for i > j (the "[64,64] WY
         matrix" that recompute_w_u takes as given; its definition is the
         reading that makes the chunked form equal the token recurrence).
  w, u   recompute_w_u: u = A (v * beta), w = A (k * beta * exp(g)).
  h      chunk_fwd_h: per chunk (1) store h, (2) v_new = u - w @ h,
         (3) v_gated = v_new * exp(g_last - g_t), (4) h *= exp(g_last),
         (5) h += k^T @ v_gated.
  o      chunk_fwd_o: scale * (q @ h * exp(g)) + causal(q @ k^T * exp(g_i - g_j)) @ v_new,
         mask i >= j, with h the state stored at step (1) and v_new the ungated
         value of step (2); scale multiplies both terms.

g is the chunk-local cumulative log-decay (restarted every C tokens). A tail
chunk (T not a multiple of C) holds only its valid rows; g_last is the g of
its last valid token. The triangular inverse uses a library triangular solve.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def _lower_gate(gc: np.ndarray, strict: bool) -> np.ndarray:
    """exp(g_i - g_j) on the (strictly) lower triangle, 0 elsewhere.

    The exponent is masked before exp is taken: above the diagonal g_i - g_j
    may be large and positive and is never evaluated."""
    n = gc.shape[0]
    i, j = np.indices((n, n))
    keep = (i > j) if strict else (i >= j)
    diff = np.where(keep, gc[:, None] - gc[None, :], -np.inf)
    return np.exp(diff)


def chunk_wy(kc, gc, bc):
    """A = (I + L)^-1 for one chunk."""
    n = kc.shape[0]
    L = (bc[:, None] * (kc @ kc.T)) * _lower_gate(gc, strict=True)
    return solve_triangular(np.eye(n) + L, np.eye(n), lower=True, unit_diagonal=True)


def forward(q, k, v, g, beta, scale=1.0, h0=None, *, chunk: int = 64, stages: bool = False):
    """Chunked forward in fp64. Arrays [B,T,H,*]; returns dict with o, h_final and,
    if ``stages``, A [B,T,H,C], w, u, v_new [B,T,H,*] and h [B,NT,H,K,V]."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    NT = (T + chunk - 1) // chunk
    o = np.zeros((B, T, H, V))
    h_final = np.zeros((B, H, K, V))
    if stages:
        A_all = np.zeros((B, T, H, chunk))
        w_all = np.zeros((B, T, H, K))
        u_all = np.zeros((B, T, H, V))
        vn_all = np.zeros((B, T, H, V))
        h_all = np.zeros((B, NT, H, K, V))
    for b in range(B):
        for hh in range(H):
            S = np.zeros((K, V)) if h0 is None else np.array(h0[b, hh], dtype=np.float64)
            for c in range(NT):
                s, e = c * chunk, min(T, (c + 1) * chunk)
                qc, kc, vc = q[b, s:e, hh], k[b, s:e, hh], v[b, s:e, hh]
                gc, bc = g[b, s:e, hh], beta[b, s:e, hh]
                A = chunk_wy(kc, gc, bc)
                u = A @ (vc * bc[:, None])
                w = A @ (kc * (bc * np.exp(gc))[:, None])
                h_c = S.copy()                                  # (1) store h
                v_new = u - w @ h_c                             # (2)
                g_last = gc[-1]
                v_gated = v_new * np.exp(g_last - gc)[:, None]  # (3)
                S = S * np.exp(g_last) + kc.T @ v_gated         # (4), (5)
                inter = (qc @ h_c) * np.exp(gc)[:, None]
                intra = ((qc @ kc.T) * _lower_gate(gc, strict=False)) @ v_new
                o[b, s:e, hh] = scale * (inter + intra)
                if stages:
                    A_all[b, s:e, hh, :e - s] = A
                    w_all[b, s:e, hh] = w
                    u_all[b, s:e, hh] = u
                    vn_all[b, s:e, hh] = v_new
                    h_all[b, c, hh] = h_c
            h_final[b, hh] = S
    out = {"o": o, "h_final": h_final}
    if stages:
        out.update(A=A_all, w=w_all, u=u_all, v_new=vn_all, h=h_all)
    return out
