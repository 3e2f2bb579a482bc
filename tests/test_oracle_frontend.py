"""The oracle's input front-end against its pins (CPU only), and planted
mistakes that the pins must catch.

Each pin takes the two front-end functions as arguments, so the same pins run
on the oracle and on broken copies of it."""
import numpy as np
import pytest

from oracle import chunked, frontend, recurrence
from tests import pins


# ----------------------------------------------------------------- l2 norm pins
def pin_norm_closed_forms(cumsum, l2norm):
    """Rows with a known sum of squares: (3, 4, 0, ..) has 25, so it maps to
    (3, 4) / sqrt(25 + 1e-6); a row of 1e-3 in one place has 1e-6, where eps
    doubles the denominator: 1e-3 / sqrt(2e-6) = sqrt(1/2); a zero row stays 0."""
    x = np.zeros((3, 8))
    x[0, :2] = (3.0, 4.0)
    x[1, 5] = 1e-3
    y = l2norm(x)
    assert np.allclose(y[0, :2], np.array([3.0, 4.0]) / np.sqrt(25.000001), rtol=1e-15, atol=0)
    assert np.all(y[0, 2:] == 0)
    assert abs(y[1, 5] - np.sqrt(0.5)) < 1e-15
    assert np.all(y[2] == 0)


def pin_norm_invariants(cumsum, l2norm):
    """Direction kept, length |x| / sqrt(|x|^2 + eps), applied to the last axis only."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 5, 3, 16)) * rng.uniform(0.01, 10.0, (2, 5, 3, 1))
    y = l2norm(x)
    n2 = np.sum(x * x, axis=-1)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.sqrt(n2 / (n2 + 1e-6)), rtol=1e-13)
    cos = np.sum(x * y, axis=-1) / (np.linalg.norm(x, axis=-1) * np.linalg.norm(y, axis=-1))
    assert np.allclose(cos, 1.0, rtol=0, atol=1e-14)


# ------------------------------------------------------------------ cumsum pins
def pin_cumsum_dyadic(cumsum, l2norm):
    """Dyadic log decays sum exactly: T = 150 over chunks of 64 restarts at 64
    and 128; each chunk's last entry is its total; the first entry of a chunk
    is that token's own decay."""
    rng = np.random.default_rng(4)
    gam = -rng.integers(0, 16, (2, 150, 3)) / 8.0
    g = cumsum(gam, 64)
    for s, e in ((0, 64), (64, 128), (128, 150)):
        assert np.array_equal(g[:, s], gam[:, s])
        assert np.array_equal(g[:, e - 1], gam[:, s:e].sum(axis=1))
        assert np.array_equal(np.diff(g[:, s:e], axis=1), gam[:, s + 1:e])


def pin_cumsum_against_per_token_recurrence(cumsum, l2norm):
    """The recurrence on cumsum(gamma) in 64-token chunks equals the recurrence
    on gamma itself in one-token chunks (where g_t is gamma_t): two readings of
    the same decays, T = 150 with a ragged tail."""
    rng = np.random.default_rng(5)
    B, T, H, K, V = 2, 150, 2, 8, 5
    q = rng.standard_normal((B, T, H, K))
    k = l2norm(rng.standard_normal((B, T, H, K)))
    v = rng.standard_normal((B, T, H, V))
    beta = rng.uniform(0.1, 1.0, (B, T, H))
    gam = -rng.uniform(0.0, 0.3, (B, T, H))
    h0 = rng.standard_normal((B, H, K, V)) * 0.1
    o1, h1 = recurrence.forward(q, k, v, cumsum(gam, 64), beta, 0.9, h0, nthreads=2)
    o2, h2 = recurrence.forward(q, k, v, gam, beta, 0.9, h0, chunk=1, nthreads=2)
    assert pins.rel(o1, o2) < 1e-12 and pins.rel(h1, h2) < 1e-12


def pin_prepared_product_form(cumsum, l2norm):
    """Unnormalised q, k and raw decays through the front-end and the chunked
    form equal the closed product form on explicitly normalised rows."""
    rng = np.random.default_rng(6)
    B, T, H, K, V, chunk = 1, 7, 2, 4, 3, 3
    q = rng.standard_normal((B, T, H, K)) * 3.0
    k = rng.standard_normal((B, T, H, K)) * 0.5
    v = rng.standard_normal((B, T, H, V))
    h0 = rng.standard_normal((B, H, K, V))
    log_alpha = -rng.uniform(0.0, 0.7, (B, T, H))
    beta = rng.uniform(0.1, 1.0, (B, T, H))
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6)
    kn = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    o_x, h_x = pins.product_form(qn, kn, v, np.exp(log_alpha), beta, 0.8, h0)
    out = chunked.forward(l2norm(q), l2norm(k), v, cumsum(log_alpha, chunk), beta, 0.8, h0,
                          chunk=chunk)
    assert pins.rel(out["o"], o_x) < 1e-12 and pins.rel(out["h_final"], h_x) < 1e-12


FRONTEND_PINS = [pin_norm_closed_forms, pin_norm_invariants, pin_cumsum_dyadic,
                 pin_cumsum_against_per_token_recurrence, pin_prepared_product_form]


@pytest.mark.parametrize("pin", FRONTEND_PINS, ids=lambda p: p.__name__)
def test_frontend_pin(pin):
    pin(frontend.chunk_cumsum, frontend.l2norm_rows)


def test_prepare_applies_what_the_flags_select():
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal((2, 1, 70, 3, 8))
    g = -rng.uniform(0, 1, (1, 70, 3))
    for raw in (False, True):
        for norm in (False, True):
            pq, pk, pg = frontend.prepare(q, k, g, raw_g=raw, qk_l2norm=norm)
            assert np.array_equal(pq, frontend.l2norm_rows(q) if norm else q)
            assert np.array_equal(pk, frontend.l2norm_rows(k) if norm else k)
            assert np.array_equal(pg, frontend.chunk_cumsum(g) if raw else g)


# ------------------------------------------------------------------- mutants
def _cumsum_no_restart(gamma, chunk=64):
    return np.cumsum(np.asarray(gamma, dtype=np.float64), axis=1)


def _cumsum_exclusive(gamma, chunk=64):
    g = frontend.chunk_cumsum(gamma, chunk)
    return g - np.asarray(gamma, dtype=np.float64)


def _cumsum_restart_65(gamma, chunk=64):
    return frontend.chunk_cumsum(gamma, chunk + 1)


def _norm_eps_outside(x, eps=1e-6):
    x = np.asarray(x, dtype=np.float64)
    return x / (np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) + eps)


def _norm_no_sqrt(x, eps=1e-6):
    x = np.asarray(x, dtype=np.float64)
    return x / (np.sum(x * x, axis=-1, keepdims=True) + eps)


def _norm_wrong_axis(x, eps=1e-6):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-2, keepdims=True) + eps)


MUTANTS = {
    "cumsum without chunk restart": (_cumsum_no_restart, frontend.l2norm_rows),
    "exclusive cumsum": (_cumsum_exclusive, frontend.l2norm_rows),
    "chunk of 65": (_cumsum_restart_65, frontend.l2norm_rows),
    "eps outside the root": (frontend.chunk_cumsum, _norm_eps_outside),
    "norm without root": (frontend.chunk_cumsum, _norm_no_sqrt),
    "norm over the wrong axis": (frontend.chunk_cumsum, _norm_wrong_axis),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_each_planted_mistake_fails_a_pin(name):
    cumsum, l2norm = MUTANTS[name]
    caught = []
    for pin in FRONTEND_PINS:
        try:
            pin(cumsum, l2norm)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught: {name}"
