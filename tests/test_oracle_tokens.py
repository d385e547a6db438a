"""Pins for the oracle's multi-token decode (``oracle.decode_tokens``).

T decode steps in one call must equal, independently of the decode step's own
code: a direct causal convolution of each channel's token sequence with the
cache as left context (numpy.convolve) followed by SiLU, then L2 normalisation
and the chunked WY / UT form of the recurrence ("GLM-5.3 deep dive", 8.2.4
step 2 and 8.2.5 Eq. 6-9, written with numpy matmuls). The final conv cache is
the last three inputs of that sequence.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle


def _problem(rng, M, T, H, d):
    D = H * d
    x = rng.standard_normal((M, T, 3, D))
    w = 0.5 * rng.standard_normal((3, D, 4))
    cache = rng.standard_normal((M, 3, 3, D))
    a = expit(rng.standard_normal((M, T, H, d)) + 2.0)
    b = expit(rng.standard_normal((M, T, H)))
    S0 = 0.1 * rng.standard_normal((M, H, d, d))
    return x, w, cache, a, b, S0


def _direct(x, w, cache, a, b, S0, scale):
    """numpy.convolve over [cache taps, tokens] + SiLU, then the chunked form."""
    M, T, _, D = x.shape
    H, d = a.shape[2], a.shape[3]
    y = np.empty_like(x)
    new_cache = np.empty_like(cache)
    for m in range(M):
        for X in range(3):
            for c in range(D):
                seq = np.concatenate([cache[m, X, :, c], x[m, :, X, c]])
                pre = np.convolve(seq, w[X, c, ::-1], mode="valid")  # taps newest-first
                y[m, :, X, c] = pre * expit(pre)
                new_cache[m, X, :, c] = seq[-3:]
    q, k, v = (y[:, :, X].reshape(M, T, H, d) for X in range(3))
    o, S = oracle.chunk_prefill(q, k, v, a, b, S0, chunk=4, scale=scale)
    return o, S, new_cache


@pytest.mark.parametrize("T", [1, 2, 3, 5, 17])
def test_tokens_equal_convolution_then_chunked_form(T):
    rng = np.random.default_rng(700 + T)
    args = _problem(rng, 2, T, 3, 4)
    o, S, c = oracle.decode_tokens(*args, scale=0.7)
    o_ref, S_ref, c_ref = _direct(*args, scale=0.7)
    np.testing.assert_array_equal(c, c_ref)
    assert np.max(np.abs(o - o_ref)) / np.max(np.abs(o_ref)) < 1e-12
    assert np.max(np.abs(S - S_ref)) / np.max(np.abs(S_ref)) < 1e-12


def test_one_token_is_the_decode_step():
    rng = np.random.default_rng(720)
    x, w, cache, a, b, S0 = _problem(rng, 2, 1, 2, 8)
    o, S, c = oracle.decode_tokens(x, w, cache, a, b, S0, scale=0.5)
    o1, S1, c1 = oracle.decode_step(x[:, 0], w, cache, a[:, 0], b[:, 0], S0, scale=0.5)
    np.testing.assert_array_equal(o[:, 0], o1)
    np.testing.assert_array_equal(S, S1)
    np.testing.assert_array_equal(c, c1)


def test_tokens_split_anywhere():
    """Processing T tokens at once or as two calls (state and cache carried)
    gives the same result: the call is a plain composition of steps."""
    rng = np.random.default_rng(730)
    x, w, cache, a, b, S0 = _problem(rng, 1, 7, 2, 4)
    o, S, c = oracle.decode_tokens(x, w, cache, a, b, S0)
    oa, Sa, ca = oracle.decode_tokens(x[:, :3], w, cache, a[:, :3], b[:, :3], S0)
    ob, Sb, cb = oracle.decode_tokens(x[:, 3:], w, ca, a[:, 3:], b[:, 3:], Sa)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, rtol=0, atol=0)
    np.testing.assert_array_equal(Sb, S)
    np.testing.assert_array_equal(cb, c)


def test_prefill_layer_is_gate_then_tokens_then_norm():
    """The layer over a prompt composes pinned pieces: for one token it is the
    fused decode step; for T tokens, the gate applied token-wise then the
    multi-token decode, then the norm."""
    rng = np.random.default_rng(740)
    M, T, H, d = 2, 5, 2, 4
    x, w, cache, _, b, S0 = _problem(rng, M, T, H, d)
    f = rng.standard_normal((M, T, H, d))
    A = rng.uniform(-1, 1, H)
    bias = rng.standard_normal(H * d)
    og = rng.standard_normal((M, T, H, d))
    nw = 1 + 0.1 * rng.standard_normal(d)
    y, S, c = oracle.prefill_layer(x, w, cache, f, A, bias, b, S0, scale=0.5, out_gate=og, norm_w=nw)
    # token by token through the fused decode step
    Sr, cr = S0, cache
    for t in range(T):
        yt, Sr, cr = oracle.decode_step_fused(x[:, t], w, cr, f[:, t], A, bias, b[:, t], Sr,
                                              scale=0.5, out_gate=og[:, t], norm_w=nw)
        np.testing.assert_allclose(y[:, t], yt, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S, Sr, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(c, cr)
