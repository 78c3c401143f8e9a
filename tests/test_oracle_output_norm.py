"""Pins for the fp64 output RMS-normalisation oracle: values the definition
fixes, computed by other routes (closed forms, invariances, a per-row loop).
Each pin takes the function as an argument and also runs against copies with
one planted mistake each, every one of which must fail at least one pin."""
import numpy as np
import pytest

from oracle.output_norm import output_rmsnorm


def rows(seed, T=5, H=3, D=8):
    r = np.random.default_rng(seed)
    # heads on very different scales, so that normalising over the wrong axis shows
    return r.standard_normal((T, H, D)) * np.array([0.01, 1.0, 300.0])[None, :, None]


def pin_constant_row_closed_form(norm):
    # o = c * 1  ->  o' = w c / sqrt(c^2 + eps)
    c, eps, D = 0.3, 0.05, 8
    w = np.arange(1, D + 1) / 4.0
    o = np.full((1, 1, D), c)
    want = w * c / np.sqrt(c * c + eps)
    assert np.allclose(norm(o, w, eps)[0, 0], want, rtol=1e-14, atol=0)


def pin_unit_rms_and_scale_invariance(norm):
    o = rows(1)
    out = norm(o, None, 0.0)
    rms = np.sqrt((out * out).mean(axis=-1))
    assert np.allclose(rms, 1.0, rtol=1e-14, atol=0)
    assert np.allclose(norm(o * 7.5, None, 0.0), out, rtol=1e-13, atol=0)


def pin_per_row_loop(norm):
    o, eps = rows(2), 1e-3
    w = np.linspace(-2, 2, 8)
    out = norm(o, w, eps)
    for t in range(o.shape[0]):
        for h in range(o.shape[1]):
            x = o[t, h]
            s = 0.0
            for v in x:
                s += v * v
            want = [w[i] * x[i] / np.sqrt(s / len(x) + eps) for i in range(len(x))]
            assert np.allclose(out[t, h], want, rtol=1e-13, atol=0)


def pin_weight_linear(norm):
    o = rows(3)
    w = np.random.default_rng(4).standard_normal(8)
    assert np.allclose(norm(o, 3 * w, 1e-6), 3 * norm(o, w, 1e-6), rtol=1e-14, atol=0)
    assert np.allclose(norm(o, np.ones(8), 1e-6), norm(o, None, 1e-6), rtol=0, atol=0)


PINS = [pin_constant_row_closed_form, pin_unit_rms_and_scale_invariance, pin_per_row_loop,
        pin_weight_linear]


@pytest.mark.parametrize("pin", PINS)
def test_pin(pin):
    pin(output_rmsnorm)


def _w(weight, d):
    return np.ones(d) if weight is None else np.asarray(weight, float)


MUTANTS = {
    "sum instead of mean": lambda o, w=None, eps=1e-6: o / np.sqrt(
        (o * o).sum(-1, keepdims=True) + eps) * _w(w, o.shape[-1]),
    "no square root": lambda o, w=None, eps=1e-6: o / (
        (o * o).mean(-1, keepdims=True) + eps) * _w(w, o.shape[-1]),
    "normalised over heads": lambda o, w=None, eps=1e-6: o / np.sqrt(
        (o * o).mean(-2, keepdims=True) + eps) * _w(w, o.shape[-1]),
    "eps outside the root": lambda o, w=None, eps=1e-6: o / (np.sqrt(
        (o * o).mean(-1, keepdims=True)) + eps) * _w(w, o.shape[-1]),
    "weight ignored": lambda o, w=None, eps=1e-6: o / np.sqrt(
        (o * o).mean(-1, keepdims=True) + eps),
    "mean of |o| instead of rms": lambda o, w=None, eps=1e-6: o / (
        np.abs(o).mean(-1, keepdims=True) + eps) * _w(w, o.shape[-1]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    bad = MUTANTS[name]
    caught = 0
    for pin in PINS:
        try:
            pin(bad)
        except AssertionError:
            caught += 1
    assert caught >= 1, f"no pin catches: {name}"
