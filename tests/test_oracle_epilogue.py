"""The oracle's gated RMSNorm against its pins (CPU only), and planted mistakes
that the pins must catch. Each pin takes the function under test."""
import numpy as np
import pytest
from scipy.special import expit

from oracle import epilogue


def pin_constant_row(fn):
    """A row of c in all V places has mean square c^2: with gate 0 (sigmoid 1/2)
    and weight 1 each entry is c / sqrt(c^2 + eps) / 2."""
    for V, c, eps in ((64, 3.0, 1e-6), (128, -0.25, 1e-5), (16, 1e-3, 1e-6)):
        o = np.full((2, V), c)
        y = fn(o, np.zeros((2, V)), np.ones(V), eps)
        assert np.allclose(y, c / np.sqrt(c * c + eps) / 2, rtol=1e-15, atol=0), (V, c)


def pin_two_channel_row(fn):
    """(3, 4) has mean square 12.5; weight (2, -1), gate (0, ln 3): sigmoid
    (1/2, 3/4), so the row is (3, -3) / sqrt(12.5 + eps)."""
    eps = 1e-6
    y = fn(np.array([[3.0, 4.0]]), np.array([[0.0, np.log(3.0)]]), np.array([2.0, -1.0]), eps)
    want = np.array([3.0, -3.0]) / np.sqrt(12.5 + eps)
    assert np.allclose(y[0], want, rtol=1e-14, atol=0)


def pin_scale_invariance(fn):
    """With eps = 0 the result does not change when a row is scaled by l > 0
    and flips sign for l < 0; the scaling is per row (per token and head)."""
    rng = np.random.default_rng(8)
    o = rng.standard_normal((3, 5, 2, 32))
    z = rng.standard_normal((3, 5, 2, 32))
    w = rng.uniform(0.5, 1.5, 32)
    lam = rng.uniform(0.1, 10.0, (3, 5, 2, 1))
    y = fn(o, z, w, 0.0)
    assert np.allclose(fn(o * lam, z, w, 0.0), y, rtol=1e-13, atol=1e-15)
    assert np.allclose(fn(-o, z, w, 0.0), -y, rtol=1e-13, atol=1e-15)


def pin_unit_rms_when_open(fn):
    """Gate far open (sigmoid = 1 to 1e-17) and weight 1: each row's mean
    square is m / (m + eps), m the input's mean square."""
    rng = np.random.default_rng(9)
    o = rng.standard_normal((4, 48)) * rng.uniform(0.01, 5.0, (4, 1))
    y = fn(o, np.full((4, 48), 40.0), np.ones(48), 1e-5)
    m = np.mean(o * o, axis=-1)
    assert np.allclose(np.mean(y * y, axis=-1), m / (m + 1e-5), rtol=1e-13)


def pin_gate_and_weight_per_channel(fn):
    """Gate and weight act channel by channel: with one row, the ratio of the
    output to the ungated, unweighted output is weight_v sigmoid(gate_v)."""
    rng = np.random.default_rng(10)
    o = rng.standard_normal((1, 24))
    z = rng.standard_normal((1, 24)) * 3
    w = rng.standard_normal(24)
    base = fn(o, np.full((1, 24), 40.0), np.ones(24), 1e-6)
    y = fn(o, z, w, 1e-6)
    assert np.allclose(y / base, w * expit(z), rtol=1e-13)


PINS = [pin_constant_row, pin_two_channel_row, pin_scale_invariance, pin_unit_rms_when_open,
        pin_gate_and_weight_per_channel]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_epilogue_pin(pin):
    pin(epilogue.gated_rmsnorm)


def _sum_not_mean(o, gate, weight, eps):
    o = np.asarray(o, dtype=np.float64)
    return o / np.sqrt(np.sum(o * o, axis=-1, keepdims=True) + eps) * weight * expit(gate)


def _eps_outside(o, gate, weight, eps):
    o = np.asarray(o, dtype=np.float64)
    return o / (np.sqrt(np.mean(o * o, axis=-1, keepdims=True)) + eps) * weight * expit(gate)


def _sigmoid_of_minus(o, gate, weight, eps):
    return epilogue.gated_rmsnorm(o, -np.asarray(gate), weight, eps)


def _no_weight(o, gate, weight, eps):
    return epilogue.gated_rmsnorm(o, gate, np.ones_like(np.asarray(weight)), eps)


def _wrong_axis(o, gate, weight, eps):
    o = np.asarray(o, dtype=np.float64)
    return o / np.sqrt(np.mean(o * o, axis=0, keepdims=True) + eps) * weight * expit(gate)


def _gate_not_squashed(o, gate, weight, eps):
    o = np.asarray(o, dtype=np.float64)
    return o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) * weight * np.asarray(gate)


MUTANTS = {"sum instead of mean": _sum_not_mean, "eps outside the root": _eps_outside,
           "sigmoid of -gate": _sigmoid_of_minus, "weight dropped": _no_weight,
           "norm over the wrong axis": _wrong_axis, "gate without sigmoid": _gate_not_squashed}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_each_planted_mistake_fails_a_pin(name):
    caught = []
    for pin in PINS:
        try:
            pin(MUTANTS[name])
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught: {name}"
