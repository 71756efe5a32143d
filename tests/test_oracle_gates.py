"""Pins for the oracle's decay / write-strength prologue (g and beta from their logits).

Reading (the pages list the parameters -- A_log = log U(1, 16) per head, a bias per
decay logit, gate_lower_bound, beta = sigmoid(b_proj) -- but omit the line that
combines them): g = max(lower_bound, -exp(A_log[h]) * softplus(z + dt_bias)),
beta = sigmoid(b).  Pinned against library routines (numpy logaddexp for softplus,
scipy expit for the sigmoid), closed forms (softplus(0) = ln 2, the clamp, the
large-logit asymptote) and planted mistakes that must each fail a pin.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle


def oracle_runner(z, A_log, b, dt_bias=None, lb=None):
    return oracle.gates(z, A_log, b, dt_bias, lb)


def mutant(kind):
    def run(z, A_log, b, dt_bias=None, lb=None):
        z = np.asarray(z, np.float64)
        x = z + (0.0 if dt_bias is None or kind == "no_bias" else np.asarray(dt_bias, np.float64))
        a = np.asarray(A_log, np.float64)[:, None]
        a = a if kind == "a_not_exp" else np.exp(a)
        sp = np.exp(x) if kind == "exp_not_softplus" else np.logaddexp(0.0, x)
        g = -a * sp
        if lb is not None:
            g = np.minimum(g, lb) if kind == "clamp_wrong_way" else np.maximum(g, lb)
        bb = np.asarray(b, np.float64)
        beta = np.tanh(bb) if kind == "tanh_beta" else scipy.special.expit(bb)
        return g, beta
    return run


def _data(seed=0, R=5, H=3, K=8):
    r = np.random.default_rng(seed)
    z = (r.standard_normal((R, H, K)) * 3 - 1).astype(np.float32)
    A_log = np.log(r.uniform(1, 16, H)).astype(np.float32)
    dtb = r.uniform(-1, 1, (H, K)).astype(np.float32)
    b = r.standard_normal((R, H)).astype(np.float32) * 2
    return z, A_log, dtb, b


def pin_library(run):
    """softplus = logaddexp(0, x) and the sigmoid = expit, in fp64."""
    z, A_log, dtb, b = _data()
    g, beta = run(z, A_log, b, dtb, None)
    x = z.astype(np.float64) + dtb
    ref = -np.exp(A_log.astype(np.float64))[:, None] * np.logaddexp(0.0, x)
    return np.allclose(g, ref, rtol=1e-13, atol=0) and np.allclose(beta, scipy.special.expit(b.astype(np.float64)),
                                                                   rtol=1e-14, atol=0)


def pin_softplus_zero(run):
    """z + bias = 0 and A_log = 0: g = -ln 2 exactly; b = 0: beta = 1/2."""
    z = np.full((2, 2, 4), 0.5, np.float32)
    dtb = np.full((2, 4), -0.5, np.float32)
    g, beta = run(z, np.zeros(2, np.float32), np.zeros((2, 2), np.float32), dtb, None)
    return np.allclose(g, -math.log(2.0), rtol=1e-15, atol=0) and np.all(beta == 0.5)


def pin_per_head_scale(run):
    """A_log = log a_h scales the head's softplus by a_h."""
    z, _, dtb, b = _data(seed=1)
    g1, _ = run(z, np.zeros(3, np.float32), b, dtb, None)
    a = np.array([1.0, 2.0, 16.0], np.float32)
    g2, _ = run(z, np.log(a), b, dtb, None)
    return np.allclose(g2, g1 * a.astype(np.float64)[:, None], rtol=1e-6, atol=0)


def pin_clamp(run):
    """The lower bound is a floor: g = max(lb, raw)."""
    z, A_log, dtb, b = _data(seed=2)
    raw, _ = run(z, A_log, b, dtb, None)
    g, _ = run(z, A_log, b, dtb, -5.0)
    return np.array_equal(g, np.maximum(raw, -5.0)) and np.any(raw < -5.0) and np.any(raw > -5.0)


def pin_asymptotes(run):
    """Large logits: softplus(x) -> x; very negative: softplus(x) -> e^x (relative)."""
    z = np.array([[[30.0, -30.0]]], np.float32)
    g, _ = run(z, np.zeros(1, np.float32), np.zeros((1, 1), np.float32), None, None)
    return abs(g[0, 0, 0] + 30.0) < 1e-12 and abs(g[0, 0, 1] + math.exp(-30.0)) < 1e-25


def pin_beta_symmetry(run):
    z, A_log, dtb, b = _data(seed=3)
    _, b1 = run(z, A_log, b, dtb, None)
    _, b2 = run(z, A_log, -b, dtb, None)
    return np.allclose(b1 + b2, 1.0, rtol=0, atol=1e-15) and np.all((b1 > 0) & (b1 < 1))


PINS = [pin_library, pin_softplus_zero, pin_per_head_scale, pin_clamp, pin_asymptotes, pin_beta_symmetry]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    assert pin(oracle_runner)


@pytest.mark.parametrize("kind", ["no_bias", "a_not_exp", "exp_not_softplus", "clamp_wrong_way", "tanh_beta"])
def test_pins_catch_mutant(kind):
    assert not all(p(mutant(kind)) for p in PINS), f"no pin catches '{kind}'"


def test_mutant_harness_is_faithful():
    assert all(p(mutant("none")) for p in PINS)


def test_gates_in_range_and_used_unrounded():
    """With the -5 floor every g lies in [-5, 0] and beta in (0, 1); the recurrence takes
    the fp64 gates as they are (rounding them to fp32 changes its output)."""
    r = np.random.default_rng(4)
    T, H, K, V = 6, 2, 8, 8
    q = r.standard_normal((1, T, H, K)).astype(np.float32)
    k = r.standard_normal((1, T, H, K)).astype(np.float32)
    v = r.standard_normal((1, T, H, V)).astype(np.float32)
    z = (r.standard_normal((1, T, H, K)) - 1).astype(np.float32)
    bl = r.standard_normal((1, T, H)).astype(np.float32)
    A_log = np.log(r.uniform(1, 16, H)).astype(np.float32)
    g, beta = oracle.gates(z, A_log, bl, None, -5.0)
    assert g.dtype == np.float64 and np.all(g <= 0) and np.all(g >= -5) and np.all((beta > 0) & (beta < 1))
    o1, _ = oracle.recurrent(q, k, v, g, beta)
    o2, _ = oracle.recurrent(q, k, v, g.astype(np.float32), beta.astype(np.float32))
    assert not np.array_equal(o1, o2) and np.allclose(o1, o2, rtol=1e-5, atol=1e-6)
