"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle.

Each ``pin_*`` takes a forward function ``fwd(q, k, v, g, beta, scale, h0, chunk)
-> (o, h_final)`` (arrays in [B,T,H,*] layout) and raises AssertionError when
the function disagrees with the pinned fact. The same pins run against the C
recurrence, the NumPy chunked form and deliberately broken copies of the C
recurrence (which must fail at least one pin).

The inputs are built from chosen per-token decays alpha_t; the g handed to the
forward is their chunk-local cumulative log (the form the chunked kernels of
the "WarpDrive" page consume), so no pin re-derives g the way the oracle does.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def g_from_log_alpha(log_alpha: np.ndarray, chunk: int) -> np.ndarray:
    """[B,T,H] per-token log-decays -> chunk-local cumulative sums (fp64)."""
    g = np.zeros_like(log_alpha, dtype=np.float64)
    T = log_alpha.shape[1]
    for s in range(0, T, chunk):
        g[:, s:s + chunk] = np.cumsum(log_alpha[:, s:s + chunk], axis=1)
    return g


# ---------------------------------------------------------------- brute force
def product_form(q, k, v, alpha, beta, scale, h0):
    """Closed product form, per sequence, recomputed from scratch for every t:

        S_t = P(t,0) h0 + sum_{j<=t} P(t,j+1) beta_j k_j v_j^T,
        P(t,s) = M_t M_{t-1} ... M_s,   M_r = alpha_r (I - beta_r k_r k_r^T),
        o_t = scale * S_t^T q_t.

    Works on float arrays or on object arrays of Fractions (exact)."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    obj = q.dtype == object
    one = Fraction(1) if obj else 1.0
    zero = Fraction(0) if obj else 0.0

    def eye(n):
        m = np.full((n, n), zero, dtype=object if obj else np.float64)
        for i in range(n):
            m[i, i] = one
        return m

    o = np.full((B, T, H, V), zero, dtype=object if obj else np.float64)
    hf = np.full((B, H, K, V), zero, dtype=object if obj else np.float64)
    for b in range(B):
        for h in range(H):
            M = []
            for r in range(T):
                kr = k[b, r, h].reshape(K, 1)
                M.append(alpha[b, r, h] * (eye(K) - beta[b, r, h] * (kr @ kr.T)))

            def P(t, s):
                acc = eye(K)
                for r in range(s, t + 1):
                    acc = M[r] @ acc
                return acc

            h0s = h0[b, h] if h0 is not None else np.full((K, V), zero, dtype=object if obj else np.float64)
            for t in range(T):
                S = P(t, 0) @ h0s
                for j in range(t + 1):
                    kj = k[b, j, h].reshape(K, 1)
                    vj = v[b, j, h].reshape(1, V)
                    S = S + P(t, j + 1) @ (beta[b, j, h] * (kj @ vj))
                o[b, t, h] = scale * (S.T @ q[b, t, h])
                if t == T - 1:
                    hf[b, h] = S
    return o, hf


def _dyadic(rng, shape, choices):
    idx = rng.integers(0, len(choices), size=shape)
    out = np.empty(shape, dtype=object)
    for pos in np.ndindex(*shape):
        out[pos] = choices[idx[pos]]
    return out


def pin_rational(fwd):
    """Exact rational arithmetic: decays alpha in {1/4,1/2,3/4,1}, dyadic q,k,v,beta,h0.
    Two chunks of 4 tokens (crosses the chunk boundary), 2 batches x 2 heads."""
    rng = np.random.default_rng(11)
    B, T, H, K, V, chunk = 2, 7, 2, 3, 2, 4
    F = Fraction
    vals = [F(-1), F(-1, 2), F(-1, 4), F(0), F(1, 4), F(1, 2), F(3, 4), F(1)]
    q = _dyadic(rng, (B, T, H, K), vals)
    k = _dyadic(rng, (B, T, H, K), vals)
    v = _dyadic(rng, (B, T, H, V), vals)
    h0 = _dyadic(rng, (B, H, K, V), vals)
    alpha = _dyadic(rng, (B, T, H), [F(1, 4), F(1, 2), F(3, 4), F(1)])
    beta = _dyadic(rng, (B, T, H), [F(1, 4), F(1, 2), F(3, 4), F(1)])
    scale = F(1, 2)
    o_x, hf_x = product_form(q, k, v, alpha, beta, scale, h0)
    fl = lambda a: np.vectorize(float)(a).astype(np.float64)
    g = g_from_log_alpha(np.log(fl(alpha)), chunk)
    o, hf = fwd(fl(q), fl(k), fl(v), g, fl(beta), float(scale), fl(h0), chunk)
    assert rel(o, fl(o_x)) < 1e-12, f"rational o: {rel(o, fl(o_x))}"
    assert rel(hf, fl(hf_x)) < 1e-12, f"rational h_final: {rel(hf, fl(hf_x))}"


def pin_product_form(fwd):
    """Random fp64 inputs against the product form, T=8 over chunks of 3."""
    rng = np.random.default_rng(12)
    B, T, H, K, V, chunk = 2, 8, 2, 4, 3, 3
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    h0 = rng.standard_normal((B, H, K, V))
    log_alpha = -rng.uniform(0.0, 0.7, (B, T, H))
    beta = rng.uniform(0.1, 1.0, (B, T, H))
    o_x, hf_x = product_form(q, k, v, np.exp(log_alpha), beta, 0.7, h0)
    o, hf = fwd(q, k, v, g_from_log_alpha(log_alpha, chunk), beta, 0.7, h0, chunk)
    assert rel(o, o_x) < 1e-12, f"product form o: {rel(o, o_x)}"
    assert rel(hf, hf_x) < 1e-12, f"product form h_final: {rel(hf, hf_x)}"


def pin_product_form_per_token(fwd):
    """Chunks of one token: g is then each token's own log-decay (the form the
    decode step takes). Random fp64 inputs against the product form, T=5."""
    rng = np.random.default_rng(13)
    B, T, H, K, V = 2, 5, 3, 4, 3
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    h0 = rng.standard_normal((B, H, K, V))
    log_alpha = -rng.uniform(0.0, 2.0, (B, T, H))
    beta = rng.uniform(0.1, 1.0, (B, T, H))
    o_x, hf_x = product_form(q, k, v, np.exp(log_alpha), beta, 1.3, h0)
    o, hf = fwd(q, k, v, log_alpha, beta, 1.3, h0, 1)
    assert rel(o, o_x) < 1e-12, f"per-token product form o: {rel(o, o_x)}"
    assert rel(hf, hf_x) < 1e-12, f"per-token product form h_final: {rel(hf, hf_x)}"


# ---------------------------------------------------------------- closed forms
def pin_beta_zero(fwd):
    """beta = 0: no writes, so S_t = exp(G_t) h0 with G_t the running sum of the
    per-token log-decays, h_final = exp(G_T) h0 and o_t = scale exp(G_t) h0^T q_t."""
    rng = np.random.default_rng(13)
    B, T, H, K, V, chunk = 2, 100, 2, 6, 5, 64
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    h0 = rng.standard_normal((B, H, K, V))
    log_alpha = -rng.uniform(0.0, 0.05, (B, T, H))
    G = np.cumsum(log_alpha, axis=1)
    o, hf = fwd(q, k, v, g_from_log_alpha(log_alpha, chunk), np.zeros((B, T, H)), 1.3, h0, chunk)
    hf_x = np.exp(G[:, -1])[:, :, None, None] * h0
    o_x = 1.3 * np.exp(G)[..., None] * np.einsum("bhkv,bthk->bthv", h0, q)
    assert rel(hf, hf_x) < 1e-12, f"beta=0 h_final: {rel(hf, hf_x)}"
    assert rel(o, o_x) < 1e-12, f"beta=0 o: {rel(o, o_x)}"


def pin_orthonormal_retrieval(fwd):
    """g = 0, beta = 1, orthonormal keys, h0 = 0: h_final = sum_j k_j v_j^T and
    h_final^T k_j = v_j (each key retrieves its value exactly, to rounding)."""
    rng = np.random.default_rng(14)
    B, T, H, K, V, chunk = 1, 16, 2, 16, 5, 64
    k = np.zeros((B, T, H, K))
    for h in range(H):
        Q, _ = np.linalg.qr(rng.standard_normal((K, K)))
        k[0, :, h] = Q.T[:T]
    v = rng.standard_normal((B, T, H, V))
    q = rng.standard_normal((B, T, H, K))
    o, hf = fwd(q, k, v, np.zeros((B, T, H)), np.ones((B, T, H)), 1.0, None, chunk)
    hf_x = np.einsum("bthk,bthv->bhkv", k, v)
    assert rel(hf, hf_x) < 1e-12, f"orthonormal h_final: {rel(hf, hf_x)}"
    got = np.einsum("bhkv,bthk->bthv", hf, k)
    assert rel(got, v) < 1e-12, f"orthonormal retrieval: {rel(got, v)}"


def pin_overwrite(fwd):
    """g = 0, beta = 1: writing (k, v1) then (k, v2) with a unit key leaves k v2^T;
    querying with q = k returns v1 after the first token and v2 after the second."""
    rng = np.random.default_rng(15)
    B, T, H, K, V, chunk = 1, 2, 1, 8, 4, 64
    kk = rng.standard_normal(K)
    kk /= np.linalg.norm(kk)
    k = np.stack([kk, kk])[None, :, None, :]
    v = rng.standard_normal((B, T, H, V))
    o, hf = fwd(k.copy(), k, v, np.zeros((B, T, H)), np.ones((B, T, H)), 1.0, None, chunk)
    assert rel(o[0, 0, 0], v[0, 0, 0]) < 1e-12, "overwrite: first read"
    assert rel(o[0, 1, 0], v[0, 1, 0]) < 1e-12, "overwrite: second read"
    assert rel(hf[0, 0], np.outer(kk, v[0, 1, 0])) < 1e-12, "overwrite: state"


def pin_forget_reset(fwd):
    """A log-decay of -1e4 at token t0 erases the state: S_t0 = beta k v^T exactly,
    so o_t0 = scale beta (k . q) v; checked at a chunk start and mid-chunk."""
    rng = np.random.default_rng(16)
    B, T, H, K, V, chunk = 1, 80, 2, 6, 5, 16
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    beta = rng.uniform(0.2, 1.0, (B, T, H))
    h0 = rng.standard_normal((B, H, K, V))
    for t0 in (32, 45):
        log_alpha = -rng.uniform(0.0, 0.1, (B, T, H))
        log_alpha[:, t0] = -1e4
        o, _ = fwd(q, k, v, g_from_log_alpha(log_alpha, chunk), beta, 0.9, h0, chunk)
        for h in range(H):
            kq = k[0, t0, h] @ q[0, t0, h]
            ref = 0.9 * beta[0, t0, h] * kq * v[0, t0, h]
            assert rel(o[0, t0, h], ref) < 1e-12, f"forget reset t0={t0}"


# ---------------------------------------------------------------- structure
def pin_split_resume(fwd):
    """fwd(T1) then fwd(T2, h0 = h_final) equals fwd(T1 + T2) when chunk | T1."""
    rng = np.random.default_rng(17)
    B, H, K, V, chunk, T1, T2 = 2, 2, 8, 6, 16, 48, 37
    T = T1 + T2
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    beta = rng.uniform(0.0, 1.0, (B, T, H))
    g = g_from_log_alpha(-rng.uniform(0, 0.2, (B, T, H)), chunk)
    h0 = rng.standard_normal((B, H, K, V))
    o, hf = fwd(q, k, v, g, beta, 1.0, h0, chunk)
    o1, hf1 = fwd(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], beta[:, :T1], 1.0, h0, chunk)
    o2, hf2 = fwd(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], beta[:, T1:], 1.0, hf1, chunk)
    assert rel(np.concatenate([o1, o2], axis=1), o) < 1e-12, "split/resume o"
    assert rel(hf2, hf) < 1e-12, "split/resume h_final"


def pin_causal_and_independent(fwd):
    """o_t depends on no token after t, and sequences (b, h) do not interact:
    changing the tail leaves earlier outputs bit-identical; swapping two heads
    swaps their outputs bit-identically."""
    rng = np.random.default_rng(18)
    B, T, H, K, V, chunk = 2, 40, 3, 5, 4, 16
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    beta = rng.uniform(0.0, 1.0, (B, T, H))
    g = g_from_log_alpha(-rng.uniform(0, 0.2, (B, T, H)), chunk)
    h0 = rng.standard_normal((B, H, K, V))
    o, hf = fwd(q, k, v, g, beta, 1.0, h0, chunk)
    t0 = 23
    q2, k2, v2, b2 = q.copy(), k.copy(), v.copy(), beta.copy()
    q2[:, t0:] += 1.0
    k2[:, t0:] -= 0.5
    v2[:, t0:] *= 3.0
    b2[:, t0:] = 0.5
    o2, _ = fwd(q2, k2, v2, g, b2, 1.0, h0, chunk)
    assert np.array_equal(o2[:, :t0], o[:, :t0]), "causality"
    assert not np.allclose(o2[:, t0:], o[:, t0:]), "causality: tail did change"
    perm = [2, 0, 1]
    o3, hf3 = fwd(q[:, :, perm], k[:, :, perm], v[:, :, perm], g[:, :, perm], beta[:, :, perm],
                  1.0, h0[:, perm], chunk)
    assert np.array_equal(o3, o[:, :, perm]), "head independence o"
    assert np.array_equal(hf3, hf[:, perm]), "head independence h_final"


ALL_PINS = [pin_rational, pin_product_form, pin_product_form_per_token, pin_beta_zero, pin_orthonormal_retrieval,
            pin_overwrite, pin_forget_reset, pin_split_resume, pin_causal_and_independent]
