"""The oracle's per-channel (KDA) decay against its pins (CPU only), and planted
mistakes in copies of the C oracle that the pins must catch.

With per-channel decay, row i of the state decays by its own factor before the
read: S_t = (I - beta_t k_t k_t^T) diag(alpha_t) S_{t-1} + beta_t k_t v_t^T."""
import numpy as np
import pytest

from oracle import recurrence
from tests import pins


def g_from_log_alpha_pc(log_alpha, chunk):
    """[B,T,H,K] per-channel log-decays -> chunk-local cumulative sums."""
    g = np.empty_like(log_alpha)
    for s in range(0, log_alpha.shape[1], chunk):
        g[:, s:s + chunk] = np.cumsum(log_alpha[:, s:s + chunk], axis=1)
    return g


def product_form_pc(q, k, v, alpha, beta, scale, h0):
    """Dense-matrix form: M_t = (I - beta_t k_t k_t^T) diag(alpha_t)."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    hf = np.zeros((B, H, K, V))
    for b in range(B):
        for h in range(H):
            S = h0[b, h].copy()
            for t in range(T):
                kt = k[b, t, h]
                M = (np.eye(K) - beta[b, t, h] * np.outer(kt, kt)) @ np.diag(alpha[b, t, h])
                S = M @ S + beta[b, t, h] * np.outer(kt, v[b, t, h])
                o[b, t, h] = scale * S.T @ q[b, t, h]
            hf[b, h] = S
    return o, hf


def _inputs(rng, B, T, H, K, V, lo=0.0, hi=0.7):
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    h0 = rng.standard_normal((B, H, K, V))
    log_alpha = -rng.uniform(lo, hi, (B, T, H, K))
    beta = rng.uniform(0.1, 1.0, (B, T, H))
    return q, k, v, h0, log_alpha, beta


def pin_pc_product_form(fwd):
    """Random fp64 inputs against the dense product form, T = 9 over chunks of 4."""
    rng = np.random.default_rng(31)
    q, k, v, h0, la, beta = _inputs(rng, 2, 9, 2, 5, 3)
    o_x, h_x = product_form_pc(q, k, v, np.exp(la), beta, 0.6, h0)
    o, hf = fwd(q, k, v, g_from_log_alpha_pc(la, 4), beta, 0.6, h0, 4)
    assert pins.rel(o, o_x) < 1e-12 and pins.rel(hf, h_x) < 1e-12


def pin_pc_beta_zero(fwd):
    """beta = 0: row i of the state is h0's row i times exp(sum of its decays)."""
    rng = np.random.default_rng(32)
    q, k, v, h0, la, beta = _inputs(rng, 1, 70, 2, 6, 4)
    o, hf = fwd(q, k, v, g_from_log_alpha_pc(la, 64), np.zeros_like(beta), 1.0, h0, 64)
    want = np.exp(la.sum(axis=1))[..., None] * h0
    assert pins.rel(hf, want) < 1e-12
    G = np.exp(np.cumsum(la, axis=1))                      # [B,T,H,K]
    o_x = np.einsum("bthk,bhkv->bthv", q * G, h0)
    assert pins.rel(o, o_x) < 1e-12


def pin_pc_channel_permutation(fwd):
    """Permuting the channels of q, k, the decays and h0's rows permutes
    h_final's rows and leaves o unchanged."""
    rng = np.random.default_rng(33)
    q, k, v, h0, la, beta = _inputs(rng, 2, 40, 2, 7, 3)
    perm = rng.permutation(7)
    g = g_from_log_alpha_pc(la, 16)
    o1, h1 = fwd(q, k, v, g, beta, 0.9, h0, 16)
    o2, h2 = fwd(q[..., perm], k[..., perm], v, g[..., perm], beta, 0.9, h0[:, :, perm], 16)
    assert pins.rel(o2, o1) < 1e-12 and pins.rel(h2, h1[:, :, perm]) < 1e-12


def pin_pc_uniform_is_scalar(fwd):
    """Equal decays in every channel give the scalar rule, itself pinned by the
    scalar pins: the per-channel run equals the scalar product form."""
    rng = np.random.default_rng(34)
    q, k, v, h0, la, beta = _inputs(rng, 2, 8, 2, 4, 3)
    la_s = la[..., 0]
    o_x, h_x = pins.product_form(q, k, v, np.exp(la_s), beta, 0.7, h0)
    g = g_from_log_alpha_pc(np.repeat(la_s[..., None], 4, axis=-1), 3)
    o, hf = fwd(q, k, v, g, beta, 0.7, h0, 3)
    assert pins.rel(o, o_x) < 1e-12 and pins.rel(hf, h_x) < 1e-12


PC_PINS = [pin_pc_product_form, pin_pc_beta_zero, pin_pc_channel_permutation,
           pin_pc_uniform_is_scalar]


def fwd_oracle(q, k, v, g, beta, scale, h0, chunk, lib=None):
    return recurrence.forward(q, k, v, g, beta, scale, h0, chunk=chunk, nthreads=2, lib=lib)


@pytest.mark.parametrize("pin", PC_PINS, ids=lambda p: p.__name__)
def test_pc_pin(pin):
    pin(fwd_oracle)


MUTANTS = {
    "channel_zero_decay_for_all": ("const double ai = exp(gamma_i);",
                                   "const double ai = exp(i == 0 ? gamma_i : gk[0]);"),
    "previous_token_wrong_row": ("j->g[(row - H) * K + i]", "j->g[(row - 1) * K + i]"),
    "neighbouring_channel": ("const double ai = exp(gamma_i);",
                             "const double ai = exp((t % j->chunk == 0) ? gk[(i + 1) % K] : "
                             "gk[(i + 1) % K] - j->g[(row - H) * K + (i + 1) % K]);"),
    "cumsum_read_as_raw": ("(t % j->chunk == 0) ? gk[i] : gk[i] - j->g[(row - H) * K + i]",
                           "gk[i]"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pc_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = recurrence.SRC.read_text()
    assert src.count(old) == 1, f"mutation site for {name} not found"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = recurrence.load(recurrence.build(force=True, src=mut, out=tmp_path / "libmutant.so"))
    caught = []
    for pin in PC_PINS:
        try:
            pin(lambda *a: fwd_oracle(*a, lib=lib))
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
