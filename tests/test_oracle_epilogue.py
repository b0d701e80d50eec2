"""Pins of the output-epilogue oracle (RMSNorm, gain, SiLU output gate).

Each pin rests on something other than the oracle's own formula: values
worked by hand, the identities of SiLU and of a root-mean-square norm, and
PyTorch's own float64 rms_norm and silu routines. The last test plants the
plausible mistakes in a copy of the oracle and checks that a pin fails on each.
"""
import math

import numpy as np
import pytest
import torch

from oracle import epilogue as ep


def _pin_hand_example(f):
    # o = [3, 4]: mean square 12.5; z = ln 3 gives sigmoid(z) = 3/4 exactly.
    o = np.array([[3.0, 4.0]])
    z = np.full((1, 2), math.log(3.0))
    w = np.array([1.0, 2.0])
    rms = math.sqrt(12.5)
    want = np.array([[3.0 / rms * 1.0, 4.0 / rms * 2.0]]) * (0.75 * math.log(3.0))
    np.testing.assert_allclose(f(o, z, w, 0.0), want, rtol=1e-14, atol=0)


def _pin_constant_row_with_eps(f):
    # a constant row c: rms = sqrt(c^2 + eps), so y = c / sqrt(c^2 + eps) w silu(z)
    c, eps = 0.5, 0.25
    o = np.full((1, 8), c)
    z = np.full((1, 8), 2.0)
    w = np.linspace(0.5, 1.5, 8)
    silu2 = 2.0 / (1.0 + math.exp(-2.0))
    want = c / math.sqrt(c * c + eps) * w * silu2
    np.testing.assert_allclose(f(o, z, w, eps)[0], want, rtol=1e-14, atol=0)


def _pin_unit_mean_square(f):
    # eps = 0, unit gain, large z (silu(z) = z to double precision): y / z has
    # mean square exactly 1 in every row, and rows are normalised independently
    rng = np.random.default_rng(7)
    o = rng.standard_normal((5, 64))
    o[2] *= 1e3
    z = np.full_like(o, 60.0)
    y = f(o, z, np.ones(64), 0.0) / 60.0
    np.testing.assert_allclose(np.mean(y * y, axis=-1), np.ones(5), rtol=1e-13)
    np.testing.assert_allclose(y[2], f(o[2:3] * 1e-3, z[2:3], np.ones(64), 0.0)[0] / 60.0,
                               rtol=1e-12)


def _pin_silu_identities(f):
    # silu(z) - silu(-z) = z and silu(0) = 0, seen through a unit row of o
    z = np.linspace(-6.0, 6.0, 49)
    o = np.ones_like(z)
    w = np.ones_like(z)
    yp = f(o[None], z[None], w, 0.0)[0]
    yn = f(o[None], -z[None], w, 0.0)[0]
    np.testing.assert_allclose(yp - yn, z, rtol=0, atol=1e-14)
    assert yp[24] == 0.0


def _pin_library(f):
    # PyTorch's float64 rms_norm (weight applied after the norm) times silu
    rng = np.random.default_rng(11)
    o = rng.standard_normal((3, 7, 128))
    z = rng.standard_normal((3, 7, 128)) * 3
    w = rng.uniform(0.5, 1.5, 128)
    eps = 1e-6
    to = torch.from_numpy
    want = torch.nn.functional.rms_norm(to(o), (128,), to(w), eps) * torch.nn.functional.silu(to(z))
    np.testing.assert_allclose(f(o, z, w, eps), want.numpy(), rtol=1e-13, atol=1e-15)


PINS = [_pin_hand_example, _pin_constant_row_with_eps, _pin_unit_mean_square,
        _pin_silu_identities, _pin_library]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__[5:])
def test_epilogue_pin(pin):
    pin(ep.rmsnorm_gate)


def _mutant(kind):
    def silu(z):
        return z / (1.0 + np.exp(-z))

    def f(o, z, w, eps):
        o, z, w = (np.asarray(a, dtype=np.float64) for a in (o, z, w))
        ms = np.mean(o * o, axis=-1, keepdims=True)
        if kind == "no_eps":
            rms = np.sqrt(ms)
        elif kind == "eps_outside_sqrt":
            rms = np.sqrt(ms) + eps
        elif kind == "sum_not_mean":
            rms = np.sqrt(np.sum(o * o, axis=-1, keepdims=True) + eps)
        elif kind == "wrong_axis":
            rms = np.sqrt(np.mean(o * o, axis=0, keepdims=True) + eps)
        else:
            rms = np.sqrt(ms + eps)
        y = o / rms
        if kind != "no_weight":
            y = y * w
        if kind == "sigmoid_gate":
            return y / (1.0 + np.exp(-z))
        if kind == "gate_before_norm":
            g = o * silu(z)
            return g / np.sqrt(np.mean(g * g, axis=-1, keepdims=True) + eps) * w
        return y * silu(z)
    return f


@pytest.mark.parametrize("kind", ["no_eps", "eps_outside_sqrt", "sum_not_mean", "wrong_axis",
                                  "no_weight", "sigmoid_gate", "gate_before_norm"])
def test_epilogue_pins_catch_planted_mistakes(kind):
    f = _mutant(kind)
    failed = 0
    for pin in PINS:
        try:
            pin(f)
        except AssertionError:
            failed += 1
    assert failed >= 1, kind
    # the unplanted copy passes every pin
    for pin in PINS:
        pin(_mutant("none"))
