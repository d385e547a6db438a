"""Pins for the oracle's forget gate and gated RMSNorm (the steps right before
and right after the KDA update in a layer), independent of their code.

Sources: "GLM-5.3 deep dive" (gangliao.me), section 8.2.3 (gate formula and
its table of keep factors) and section 8.2.4 (gated RMSNorm on the output).
"""
import math
import os

import numpy as np
import pytest
from scipy.special import expit, logit

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "forget_gate_table.txt")


def _table():
    rows, neutral, floor = [], None, None
    for line in open(GOLDEN):
        t = line.split("#")[0].split()
        if not t:
            continue
        if t[0] == "row":
            rows.append(tuple(float(v) for v in t[1:]))
        elif t[0] == "neutral":
            neutral = (float(t[1]), float(t[2]))
        elif t[0] == "floor":
            floor = float(t[1])
    return rows, neutral, floor


def _gate_at(z, A=0.0, H=1, dk=1):
    """alpha for pre-activation f + b = z (b = 0), A_log = A."""
    f = np.full((1, H, dk), z)
    return oracle.forget_gate(f, np.full(H, A), np.zeros(H * dk))[0, 0, 0]


def test_gate_table_keep_factors_and_half_lives():
    rows, _, _ = _table()
    for alpha, half_life, s in rows:
        a = _gate_at(logit(s))
        assert abs(a - alpha) < 1e-4, (a, alpha)
        # the page prints half-lives rounded: "about 69", 693, 6,931
        assert abs(math.log(0.5) / math.log(a) - half_life) / half_life < 0.01


def test_gate_neutral_point_and_floor():
    _, (g_neutral, a_neutral), a_floor = _table()
    a = _gate_at(0.0)
    assert abs(math.log(a) - g_neutral) < 1e-12
    assert abs(a - a_neutral) < 5e-4
    assert abs(_gate_at(60.0) - a_floor) < 1e-4     # sigmoid -> 1
    assert abs(_gate_at(-60.0) - 1.0) < 1e-12       # sigmoid -> 0: no forgetting


def test_gate_exp_A_scales_the_preactivation():
    """exp(A_h) multiplies f + b: A = ln 2 at z equals A = 0 at 2 z."""
    rng = np.random.default_rng(21)
    for z in rng.standard_normal(5):
        assert abs(_gate_at(z, A=math.log(2.0)) - _gate_at(2.0 * z)) < 1e-14


def test_gate_bias_per_head_and_channel():
    """f = -b cancels the bias channel by channel, whatever A is."""
    rng = np.random.default_rng(22)
    H, dk = 3, 5
    b = rng.standard_normal(H * dk)
    A = rng.standard_normal(H)
    f = -b.reshape(1, H, dk).repeat(2, axis=0)
    a = oracle.forget_gate(f, A, b)
    np.testing.assert_allclose(a, np.exp(-2.5), rtol=1e-14)


def test_gate_range():
    """alpha lies in (e^-5, 1); in floating point the sigmoid saturates, so the
    ends can be reached exactly, never crossed."""
    rng = np.random.default_rng(23)
    a = oracle.forget_gate(3 * rng.standard_normal((4, 3, 16)), rng.standard_normal(3),
                           rng.standard_normal(48))
    assert np.all(a >= math.exp(-5.0) * (1 - 1e-15)) and np.all(a <= 1.0)
    assert np.all(a > 0.0)


def test_norm_constant_vector_and_open_gate():
    """o = c (constant), gate wide open, w = 1, eps = 0: y = sign(c)."""
    o = np.full((1, 2, 8), -3.5)
    y = oracle.gated_rmsnorm(o, np.full(o.shape, 60.0), np.ones(8), eps=0.0)
    np.testing.assert_allclose(y, -1.0, rtol=1e-14)


def test_norm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(24)
    o = rng.standard_normal((2, 3, 16))
    g = rng.standard_normal((2, 3, 16))
    w = rng.standard_normal(16)
    y1 = oracle.gated_rmsnorm(o, g, w, eps=0.0)
    y2 = oracle.gated_rmsnorm(7.25 * o, g, w, eps=0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-13)
    z = y1 / (w * expit(g))
    np.testing.assert_allclose(np.mean(z * z, axis=-1), 1.0, rtol=1e-13)


def test_norm_gate_zero_halves_and_heads_independent():
    rng = np.random.default_rng(25)
    o = rng.standard_normal((1, 2, 8))
    w = np.ones(8)
    y_open = oracle.gated_rmsnorm(o, np.full(o.shape, 60.0), w)
    y_half = oracle.gated_rmsnorm(o, np.zeros(o.shape), w)
    np.testing.assert_allclose(y_half, 0.5 * y_open, rtol=1e-12)
    o2 = o.copy()
    o2[0, 1] *= -4.0
    y2 = oracle.gated_rmsnorm(o2, np.zeros(o.shape), w)
    np.testing.assert_array_equal(y2[0, 0], y_half[0, 0])


def test_norm_eps_inside_root():
    """The eps of the gated RMSNorm sits inside the root (FusedRMSNormGated,
    eps 1e-5, "GLM-5.3 deep dive" 8.2.4 notes). A constant vector o = c has
    mean(o^2) = c^2, so it normalises to c / sqrt(c^2 + eps): with c^2 = eps
    that is 1/sqrt(2), with c^2 = 3 eps it is sqrt(3)/2. The output gate at
    0 gives sigmoid(0) = 1/2 exactly and w = 1. With eps outside the root,
    c / (|c| + eps), both would be within 0.4 % of 1/2 instead: 41 % off the
    first value and 15 % off the second."""
    eps = oracle.NORM_EPS
    for c2, want in ((eps, 0.5 / math.sqrt(2.0)), (3.0 * eps, 0.25 * math.sqrt(3.0))):
        for sign in (1.0, -1.0):
            o = np.full((1, 1, 128), sign * math.sqrt(c2))
            y = oracle.gated_rmsnorm(o, np.zeros(o.shape), np.ones(128), eps=eps)
            np.testing.assert_allclose(y, sign * want, rtol=1e-12)


def test_norm_eps_keeps_zero_finite():
    y = oracle.gated_rmsnorm(np.zeros((1, 1, 8)), np.zeros((1, 1, 8)), np.ones(8))
    assert np.all(y == 0.0)


def test_fused_is_gate_then_decode_then_norm():
    from linear_attention_decode_step_gb300 import inputs
    inp = inputs.decode_layer(31, M=2, H=3, T=1)
    rng = np.random.default_rng(26)
    f = rng.standard_normal((2, 3, 128))
    A = rng.standard_normal(3)
    b = rng.standard_normal(3 * 128)
    g = rng.standard_normal((2, 3, 128))
    w = rng.standard_normal(128)
    y, S, c = oracle.decode_step_fused(inp["x_f32"][0], inp["conv_w"], inp["cache_f32"], f, A, b,
                                       inp["beta"][0], inp["S0"], out_gate=g, norm_w=w)
    alpha = oracle.forget_gate(f, A, b)
    o, S2, c2 = oracle.decode_step(inp["x_f32"][0], inp["conv_w"], inp["cache_f32"], alpha,
                                   inp["beta"][0], inp["S0"])
    np.testing.assert_array_equal(S, S2)
    np.testing.assert_allclose(y, oracle.gated_rmsnorm(o, g, w), rtol=1e-14)
