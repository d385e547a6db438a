"""Pins for the CPU oracle, independent of its own code.

Each test checks the oracle against something the pages or the mathematics
fix: the worked example of the delta rule, an explicit dense-matrix product of
Eq. 1, invariants of the update, a direct causal convolution, and the chunked
WY form reproducing the sequential recurrence. Sources: "GLM-5.3 deep dive"
(gangliao.me) sections 8.2.2, 8.2.3, 8.2.5, 8.2.6.
"""
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "delta_rule_worked_example.txt")


def _golden():
    writes, reads, halves = [], [], []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            vals = [float(t) for t in line[1:]]
            {"write": writes, "read": reads, "half": halves}[line[0]].append(vals)
    return writes, reads, halves


def _example_run(keys, values, queries, betas):
    T = len(keys)
    q = np.array(queries, dtype=np.float64).reshape(1, T, 1, 2)
    k = np.array(keys, dtype=np.float64).reshape(1, T, 1, 2)
    v = np.array(values, dtype=np.float64).reshape(1, T, 1, 1)
    a = np.ones((1, T, 1, 2))
    b = np.array(betas, dtype=np.float64).reshape(1, T, 1)
    return oracle.recurrent(q, k, v, a, b, np.zeros((1, 1, 2, 1)), use_l2norm=False)


# --------------------------------------------------------------------------
# worked example (section 8.2.2)
# --------------------------------------------------------------------------

def test_worked_example_states():
    writes, _, _ = _golden()
    for n in range(1, len(writes) + 1):
        rows = writes[:n]
        _, S = _example_run([r[1:3] for r in rows], [r[3] for r in rows],
                            [r[1:3] for r in rows], [1.0] * n)
        np.testing.assert_allclose(S[0, 0, :, 0], rows[-1][4:6], rtol=0, atol=1e-12)


def test_worked_example_reads():
    writes, reads, _ = _golden()
    for after, q0, q1, expect in reads:
        n = int(after)
        rows = writes[:n]
        queries = [r[1:3] for r in rows]
        queries[-1] = [q0, q1]          # read with the stated query at the last step
        o, _ = _example_run([r[1:3] for r in rows], [r[3] for r in rows],
                            queries, [1.0] * n)
        assert abs(o[0, -1, 0, 0] - expect) < 1e-12


def test_worked_example_half_beta():
    writes, _, halves = _golden()
    for step, beta, s0, s1 in halves:
        n = int(step)
        rows = writes[:n]
        betas = [1.0] * n
        betas[-1] = beta
        _, S = _example_run([r[1:3] for r in rows], [r[3] for r in rows],
                            [r[1:3] for r in rows], betas)
        np.testing.assert_allclose(S[0, 0, :, 0], [s0, s1], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# brute force: Eq. 1 as an explicit dense product (section 8.2.3)
# --------------------------------------------------------------------------

def _rand_problem(rng, M, T, H, dk, dv):
    q = rng.standard_normal((M, T, H, dk))
    k = rng.standard_normal((M, T, H, dk))
    v = rng.standard_normal((M, T, H, dv))
    a = expit(rng.standard_normal((M, T, H, dk)) + 2.0)
    b = expit(rng.standard_normal((M, T, H)))
    S0 = 0.1 * rng.standard_normal((M, H, dk, dv))
    return q, k, v, a, b, S0


@pytest.mark.parametrize("dk,dv", [(1, 1), (2, 3), (3, 2), (4, 4), (8, 3), (3, 8), (8, 8)])
def test_brute_force_dense_product(dk, dv):
    rng = np.random.default_rng(100 + 10 * dk + dv)
    M, T, H = 2, 5, 3
    scale = 0.7
    q, k, v, a, b, S0 = _rand_problem(rng, M, T, H, dk, dv)
    o, S = oracle.recurrent(q, k, v, a, b, S0, scale=scale, eps=0.0)
    for m in range(M):
        for h in range(H):
            St = S0[m, h].copy()
            for t in range(T):
                kh = k[m, t, h] / np.linalg.norm(k[m, t, h])
                qh = q[m, t, h] / np.linalg.norm(q[m, t, h])
                A = (np.eye(dk) - b[m, t, h] * np.outer(kh, kh)) @ np.diag(a[m, t, h])
                St = A @ St + b[m, t, h] * np.outer(kh, v[m, t, h])
                np.testing.assert_allclose(o[m, t, h], scale * (St.T @ qh),
                                           rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(S[m, h], St, rtol=1e-12, atol=1e-12)


def test_l2norm_eps_inside_root():
    """q is normalised as q / sqrt(|q|^2 + eps): with alpha=1, beta=0, S=I the
    readout returns exactly that vector."""
    rng = np.random.default_rng(7)
    d, eps = 4, 0.25
    q = rng.standard_normal((1, 1, 1, d))
    z = np.zeros((1, 1, 1, d))
    o, _ = oracle.recurrent(q, z + 1.0, z, np.ones((1, 1, 1, d)), np.zeros((1, 1, 1)),
                            np.eye(d).reshape(1, 1, d, d), eps=eps)
    np.testing.assert_allclose(o[0, 0, 0], q[0, 0, 0] / np.sqrt(np.sum(q ** 2) + eps),
                               rtol=1e-14)


# --------------------------------------------------------------------------
# invariants (sections 8.2.2 and 8.2.3)
# --------------------------------------------------------------------------

def test_alpha1_beta0_leaves_state_and_reads_it():
    rng = np.random.default_rng(1)
    q, k, v, a, b, S0 = _rand_problem(rng, 2, 3, 2, 6, 5)
    o, S = oracle.recurrent(q, k, v, np.ones_like(a), np.zeros_like(b), S0, eps=0.0)
    np.testing.assert_array_equal(S, S0)
    qh = q / np.linalg.norm(q, axis=-1, keepdims=True)
    np.testing.assert_allclose(o, np.einsum("mhij,mthi->mthj", S0, qh), rtol=1e-12, atol=1e-15)


def test_beta1_unit_key_reads_back_value():
    """beta = 1 and |k| = 1: querying with k after the step returns v exactly,
    whatever the fade did (section 8.2.3)."""
    rng = np.random.default_rng(2)
    q, k, v, a, b, S0 = _rand_problem(rng, 2, 1, 3, 7, 5)
    o, S = oracle.recurrent(k, k, v, a, np.ones_like(b), S0, eps=0.0)
    np.testing.assert_allclose(o[:, 0], v[:, 0], rtol=1e-12, atol=1e-12)
    kh = k[:, 0] / np.linalg.norm(k[:, 0], axis=-1, keepdims=True)
    np.testing.assert_allclose(np.einsum("mhij,mhi->mhj", S, kh), v[:, 0],
                               rtol=1e-12, atol=1e-12)


def test_beta0_fades_each_row_by_its_alpha():
    rng = np.random.default_rng(3)
    q, k, v, a, b, S0 = _rand_problem(rng, 1, 1, 2, 5, 4)
    _, S = oracle.recurrent(q, k, v, a, np.zeros_like(b), S0)
    np.testing.assert_allclose(S, a[:, 0, :, :, None] * S0, rtol=1e-15)


def test_erase_shrinks_only_along_key():
    """alpha = 1, v = 0: S' = (I - beta k k^T) S. The component along k shrinks
    by (1 - beta); the orthogonal part is untouched; |S'|_F <= |S|_F."""
    rng = np.random.default_rng(4)
    q, k, v, a, b, S0 = _rand_problem(rng, 1, 1, 3, 6, 4)
    _, S = oracle.recurrent(q, k, np.zeros_like(v), np.ones_like(a), b, S0, eps=0.0)
    for h in range(3):
        kh = k[0, 0, h] / np.linalg.norm(k[0, 0, h])
        np.testing.assert_allclose(kh @ S[0, h], (1 - b[0, 0, h]) * (kh @ S0[0, h]),
                                   rtol=1e-12, atol=1e-14)
        P = np.eye(6) - np.outer(kh, kh)
        np.testing.assert_allclose(P @ S[0, h], P @ S0[0, h], rtol=1e-12, atol=1e-14)
        assert np.linalg.norm(S[0, h]) <= np.linalg.norm(S0[0, h]) + 1e-15


def test_scale_is_linear_on_output_only():
    rng = np.random.default_rng(5)
    args = _rand_problem(rng, 1, 4, 2, 5, 5)
    o1, S1 = oracle.recurrent(*args, scale=1.0)
    o2, S2 = oracle.recurrent(*args, scale=0.125)
    np.testing.assert_array_equal(S1, S2)
    np.testing.assert_allclose(o2, 0.125 * o1, rtol=1e-14, atol=1e-16)


# --------------------------------------------------------------------------
# short convolution (section 8.2.4 step 2; weight [8192, 1, 4], 3 taps)
# --------------------------------------------------------------------------

def test_conv_identity_weights_is_silu():
    rng = np.random.default_rng(6)
    M, D = 2, 16
    x = rng.standard_normal((M, 3, D))
    w = np.zeros((3, D, 4))
    w[..., 3] = 1.0
    y, _ = oracle.conv_step(x, w, rng.standard_normal((M, 3, 3, D)))
    np.testing.assert_allclose(y, x * expit(x), rtol=1e-14)


def test_conv_matches_direct_causal_convolution():
    rng = np.random.default_rng(8)
    M, D, T = 2, 12, 9
    w = 0.5 * rng.standard_normal((3, D, 4))
    cache0 = rng.standard_normal((M, 3, 3, D))
    xs = rng.standard_normal((T, M, 3, D))
    cache = cache0
    ys = []
    for t in range(T):
        y, cache = oracle.conv_step(xs[t], w, cache)
        ys.append(y)
    for m in range(M):
        for X in range(3):
            for c in range(D):
                seq = np.concatenate([cache0[m, X, :, c], xs[:, m, X, c]])
                # np.convolve flips its kernel: feed the taps newest-first
                full = np.convolve(seq, w[X, c, ::-1], mode="valid")
                pre = full[:T]
                got = np.array([ys[t][m, X, c] for t in range(T)])
                np.testing.assert_allclose(got, pre * expit(pre), rtol=1e-12, atol=1e-14)
            # after T >= 3 steps the cache holds exactly the last 3 inputs
            np.testing.assert_array_equal(cache[m, X], xs[T - 3:, m, X, :])


def test_decode_step_is_conv_then_normalised_recurrence():
    rng = np.random.default_rng(9)
    M, H, d = 2, 3, 4
    D = H * d
    x = rng.standard_normal((M, 3, D))
    w = 0.5 * rng.standard_normal((3, D, 4))
    cache = rng.standard_normal((M, 3, 3, D))
    a = expit(rng.standard_normal((M, H, d)) + 2)
    b = expit(rng.standard_normal((M, H)))
    S0 = 0.1 * rng.standard_normal((M, H, d, d))
    o, S, c_new = oracle.decode_step(x, w, cache, a, b, S0, scale=0.5)
    y, c_ref = oracle.conv_step(x, w, cache)
    q, k, v = (y[:, X].reshape(M, 1, H, d) for X in range(3))
    o_ref, S_ref = oracle.recurrent(q, k, v, a[:, None], b[:, None], S0, scale=0.5)
    np.testing.assert_array_equal(c_new, c_ref)
    np.testing.assert_allclose(o, o_ref[:, 0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S, S_ref, rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------------
# chunked WY / UT form (section 8.2.5, Eq. 6-9) reproduces T sequential steps
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("C", [16, 32, 64])
def test_chunked_equals_sequential(T, C):
    rng = np.random.default_rng(1000 + T + C)
    args = _rand_problem(rng, 1, T, 2, 16, 12)
    o_seq, S_seq = oracle.recurrent(*args, scale=0.3)
    o_chk, S_chk = oracle.chunk_prefill(*args, chunk=C, scale=0.3)
    so, ss = np.max(np.abs(o_seq)), np.max(np.abs(S_seq))
    assert np.max(np.abs(o_chk - o_seq)) / so < 1e-12
    assert np.max(np.abs(S_chk - S_seq)) / ss < 1e-12


def test_chunked_equals_sequential_at_gate_floor():
    """alpha near the e^-5 gate floor (section 8.2.3) over a full 64-token
    chunk: the summed log-decay reaches about -320, still finite in float64."""
    rng = np.random.default_rng(11)
    q, k, v, a, b, S0 = _rand_problem(rng, 1, 130, 2, 8, 8)
    a = np.exp(-5.0 + 0.01 * rng.random(a.shape))
    o_seq, S_seq = oracle.recurrent(q, k, v, a, b, S0)
    o_chk, S_chk = oracle.chunk_prefill(q, k, v, a, b, S0, chunk=64)
    assert np.max(np.abs(o_chk - o_seq)) / np.max(np.abs(o_seq)) < 1e-10
    assert np.max(np.abs(S_chk - S_seq)) / np.max(np.abs(S_seq)) < 1e-10
