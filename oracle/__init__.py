"""KDA oracle — TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 CPU statement of what the KDA decode step and the
chunked prefill compute. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with the CUDA library and never imports it; both sides take their inputs from
``linear_attention_decode_step_gb300.inputs``.

Two parts:

* ``kda_oracle.c`` (loaded through ctypes): the short conv + SiLU and the
  sequential recurrence, in the order of the pages' four decode steps
  ("GLM-5.3 deep dive", 8.2.3 Eq. 1 and 8.2.6).
* ``chunk_prefill`` below (numpy): the chunkwise-parallel WY / UT form of the
  same recurrence ("GLM-5.3 deep dive", 8.2.5, Eq. 6-9), written step by step
  in the page's order with numpy matmuls as the only library primitive.

Every function is pinned by tests that do not reuse its code; nothing here is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = [
    "build",
    "conv_step",
    "recurrent",
    "decode_step",
    "chunk_prefill",
    "forget_gate",
    "gated_rmsnorm",
    "decode_step_fused",
    "decode_tokens",
    "prefill_layer",
    "L2_EPS",
    "GATE_LOWER_BOUND",
    "NORM_EPS",
]

#: eps inside the root of the L2 normalisation ("GLM-5.3 deep dive", 8.2.6,
#: implementation notes: epsilon 1e-6)
L2_EPS = 1e-6
#: lower bound of the forget gate, log-space ("GLM-5.3 deep dive", 8.2.3)
GATE_LOWER_BOUND = -5.0
#: eps of the gated RMSNorm on the output ("GLM-5.3 deep dive", 8.2.4 notes)
NORM_EPS = 1e-5

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_SO = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into libkda_oracle.so next to it (plain gcc)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(ctypes.c_double)
    I, Dd = ctypes.c_int, ctypes.c_double
    lib.kda_oracle_conv_step.argtypes = [P, P, P, P, I, I]
    lib.kda_oracle_recurrent.argtypes = [P, P, P, P, P, P, P,
                                         I, I, I, I, I, Dd, I, Dd]
    lib.kda_oracle_decode_step.argtypes = [P, P, P, P, P, P, P,
                                           I, I, I, Dd, Dd]
    lib.kda_oracle_forget_gate.argtypes = [P, P, P, Dd, P, I, I, I]
    lib.kda_oracle_gated_rmsnorm.argtypes = [P, P, P, Dd, P, I, I, I]
    for f in (lib.kda_oracle_conv_step, lib.kda_oracle_recurrent,
              lib.kda_oracle_decode_step, lib.kda_oracle_forget_gate,
              lib.kda_oracle_gated_rmsnorm):
        f.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def _f64(a) -> np.ndarray:
    return np.array(a, dtype=np.float64, order="C", copy=True)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def conv_step(x, w, cache):
    """Short conv + SiLU for one token.

    x [M,3,D], w [3,D,4], cache [M,3,3,D] -> (y [M,3,D], new cache).
    Inputs are not modified.
    """
    x, w, cache = _f64(x), _f64(w), _f64(cache)
    M, three, D = x.shape
    assert three == 3 and w.shape == (3, D, 4) and cache.shape == (M, 3, 3, D)
    y = np.empty_like(x)
    _load().kda_oracle_conv_step(_p(x), _p(w), _p(cache), _p(y), M, D)
    return y, cache


def recurrent(q, k, v, alpha, beta, S0, scale=1.0, use_l2norm=True, eps=L2_EPS):
    """Sequential KDA recurrence over T tokens.

    q, k, alpha [M,T,H,dk]; v [M,T,H,dv]; beta [M,T,H]; S0 [M,H,dk,dv]
    -> (o [M,T,H,dv], S [M,H,dk,dv]). Inputs are not modified.
    """
    q, k, v, alpha, beta, S = (_f64(a) for a in (q, k, v, alpha, beta, S0))
    M, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and alpha.shape == q.shape
    assert v.shape == (M, T, H, dv) and beta.shape == (M, T, H)
    assert S.shape == (M, H, dk, dv)
    o = np.empty((M, T, H, dv), dtype=np.float64)
    _load().kda_oracle_recurrent(_p(q), _p(k), _p(v), _p(alpha), _p(beta),
                                 _p(S), _p(o), M, T, H, dk, dv, float(scale),
                                 1 if use_l2norm else 0, float(eps))
    return o, S


def decode_step(x, w, cache, alpha, beta, S0, scale=1.0, eps=L2_EPS):
    """One fused decode step of a KDA layer (conv + SiLU, L2 norm, Eq. 1, read).

    x [M,3,D]; w [3,D,4]; cache [M,3,3,D]; alpha [M,H,d]; beta [M,H];
    S0 [M,H,d,d] -> (o [M,H,d], S [M,H,d,d], cache [M,3,3,D]).
    """
    x, w, cache, alpha, beta, S = (_f64(a) for a in (x, w, cache, alpha, beta, S0))
    M, H, d, d2 = S.shape
    assert d == d2 and x.shape == (M, 3, H * d) and alpha.shape == (M, H, d)
    assert beta.shape == (M, H) and cache.shape == (M, 3, 3, H * d)
    o = np.empty((M, H, d), dtype=np.float64)
    _load().kda_oracle_decode_step(_p(x), _p(w), _p(cache), _p(alpha), _p(beta),
                                   _p(S), _p(o), M, H, d, float(scale), float(eps))
    return o, S, cache


def forget_gate(f, A_log, dt_bias, lb=GATE_LOWER_BOUND):
    """alpha = exp(lb * sigmoid(exp(A_h) (f + b_{h,c}))).

    f [M,H,dk] (or [M,T,H,dk] flattened the same way), A_log [H],
    dt_bias [H*dk] -> alpha, same shape as f."""
    f, A_log, dt_bias = _f64(f), _f64(A_log), _f64(dt_bias)
    shape = f.shape
    H, dk = shape[-2], shape[-1]
    M = int(np.prod(shape[:-2]))
    assert A_log.shape == (H,) and dt_bias.shape == (H * dk,)
    alpha = np.empty_like(f)
    _load().kda_oracle_forget_gate(_p(f), _p(A_log), _p(dt_bias), float(lb), _p(alpha), M, H, dk)
    return alpha


def gated_rmsnorm(o, gate, w, eps=NORM_EPS):
    """y = o / sqrt(mean(o^2) + eps) * w * sigmoid(gate), per head over dv.

    o, gate [..., H, dv]; w [dv] -> y, same shape as o."""
    o, gate, w = _f64(o), _f64(gate), _f64(w)
    shape = o.shape
    H, dv = shape[-2], shape[-1]
    M = int(np.prod(shape[:-2]))
    assert gate.shape == shape and w.shape == (dv,)
    y = np.empty_like(o)
    _load().kda_oracle_gated_rmsnorm(_p(o), _p(gate), _p(w), float(eps), _p(y), M, H, dv)
    return y


def decode_step_fused(x, w, cache, f, A_log, dt_bias, beta, S0, scale=1.0,
                      out_gate=None, norm_w=None, lb=GATE_LOWER_BOUND, eps=L2_EPS,
                      norm_eps=NORM_EPS):
    """Decode step with the forget gate in front and, if out_gate is given,
    the gated RMSNorm behind: alpha = forget_gate(f), then decode_step, then
    y = gated_rmsnorm(o). Returns (y or o, S, cache)."""
    alpha = forget_gate(f, A_log, dt_bias, lb)
    o, S, cache = decode_step(x, w, cache, alpha, beta, S0, scale=scale, eps=eps)
    if out_gate is not None:
        o = gated_rmsnorm(o, out_gate, norm_w, norm_eps)
    return o, S, cache


def decode_tokens(x, w, cache, alpha, beta, S0, scale=1.0, eps=L2_EPS):
    """T consecutive decode steps of one KDA layer in one call (the
    fused-recurrent mode of "GLM-5.3 deep dive" 8.2.5, used when a few tokens
    arrive at once, e.g. to verify drafted tokens): the decode step above,
    applied to tokens t = 0 .. T-1 in order, each one seeing the conv cache
    and the state the previous one left.

    x [M,T,3,D]; w [3,D,4]; cache [M,3,3,D]; alpha [M,T,H,d]; beta [M,T,H];
    S0 [M,H,d,d] -> (o [M,T,H,d], S [M,H,d,d], cache [M,3,3,D]).
    """
    x, alpha, beta = _f64(x), _f64(alpha), _f64(beta)
    M, T = x.shape[:2]
    S, c = _f64(S0), _f64(cache)
    o = np.empty(alpha.shape[:3] + (S.shape[-1],), dtype=np.float64)
    for t in range(T):
        o[:, t], S, c = decode_step(x[:, t], w, c, alpha[:, t], beta[:, t], S,
                                    scale=scale, eps=eps)
    return o, S, c


def prefill_layer(x, w, cache, f, A_log, dt_bias, beta, S0, scale=1.0, out_gate=None,
                  norm_w=None, lb=GATE_LOWER_BOUND, eps=L2_EPS, norm_eps=NORM_EPS):
    """A KDA layer over a prompt of T tokens ("GLM-5.3 deep dive" 8.2.4):
    the forget gate turns the raw gate input f into alpha (8.2.3), then the T
    tokens go through the decode steps in order (short conv + SiLU with the
    cache as left context, L2 norm, Eq. 1, read; 8.2.5 states that the chunked
    form reaches the same result), then, if out_gate is given, the gated
    RMSNorm on each token's output (8.2.4 step 7).

    x [M,T,3,D]; w [3,D,4]; cache [M,3,3,D]; f [M,T,H,d]; A_log [H];
    dt_bias [H*d]; beta [M,T,H]; S0 [M,H,d,d]; out_gate [M,T,H,d] or None
    -> (y or o [M,T,H,d], S, cache)."""
    alpha = forget_gate(f, A_log, dt_bias, lb)
    o, S, c = decode_tokens(x, w, cache, alpha, beta, S0, scale=scale, eps=eps)
    if out_gate is not None:
        o = gated_rmsnorm(o, out_gate, norm_w, norm_eps)
    return o, S, c


def _l2norm_rows(x, eps):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def _unit_lower_solve(A, B):
    """X = (I + A)^{-1} B for strictly lower-triangular A, by forward
    substitution, one row after another (the page's UT-transform inverse)."""
    X = np.array(B, dtype=np.float64, copy=True)
    for r in range(X.shape[0]):
        X[r] -= A[r, :r] @ X[:r]
    return X


def chunk_prefill(q, k, v, alpha, beta, S0, chunk=64, scale=1.0,
                  use_l2norm=True, eps=L2_EPS):
    """Chunkwise-parallel (WY / UT transform) KDA prefill, float64.

    Follows "GLM-5.3 deep dive", 8.2.5, per chunk of C tokens with incoming
    state S and, per key channel, the cumulative log-decay G (inclusive:
    G_r = sum_{m<=r} log alpha_m, so Gamma = exp(G)):
      Eq. 6: M = (I + StrictTril(Diag(beta) (Gamma*K) (K/Gamma)^T))^{-1} Diag(beta)
      Eq. 7: W = M (Gamma*K),  U = M V
      Eq. 8: S_next = Diag(gamma^C) S + (Gamma^{i->C} * K)^T (U - W S)
      Eq. 9: O = (Gamma*Q) S + Tril((Gamma*Q)(K/Gamma)^T) (U - W S)
    where gamma^C = exp(G_C) and Gamma^{i->C} = exp(G_C - G_i).

    Domain: exp(+-G) must stay finite in float64, i.e. the summed log-decay
    over one chunk must stay above about -700 per channel.

    Shapes as in ``recurrent``; returns (o, S).
    """
    q, k, v, alpha, beta, S = (_f64(a) for a in (q, k, v, alpha, beta, S0))
    M, T, H, dk = q.shape
    dv = v.shape[-1]
    if use_l2norm:
        q, k = _l2norm_rows(q, eps), _l2norm_rows(k, eps)
    o = np.zeros((M, T, H, dv), dtype=np.float64)
    for m in range(M):
        for h in range(H):
            Sh = S[m, h]
            for c0 in range(0, T, chunk):
                c1 = min(c0 + chunk, T)
                Q, K, V = q[m, c0:c1, h], k[m, c0:c1, h], v[m, c0:c1, h]
                b = beta[m, c0:c1, h]
                G = np.cumsum(np.log(alpha[m, c0:c1, h]), axis=0)
                Kd = np.exp(G) * K          # Gamma (.) K
                Ki = K * np.exp(-G)         # K / Gamma
                Qd = np.exp(G) * Q          # Gamma (.) Q
                A = np.tril(b[:, None] * (Kd @ Ki.T), -1)
                Mx = _unit_lower_solve(A, np.diag(b))
                W, U = Mx @ Kd, Mx @ V
                Delta = U - W @ Sh
                o[m, c0:c1, h] = scale * (Qd @ Sh + np.tril(Qd @ Ki.T) @ Delta)
                Sh = np.exp(G[-1])[:, None] * Sh + (np.exp(G[-1] - G) * K).T @ Delta
            S[m, h] = Sh
    return o, S
