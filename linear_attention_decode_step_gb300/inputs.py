"""Seeded synthetic inputs for the KDA decode step and the chunked prefill.

This module only draws random numbers and packs them into the storage formats
the library consumes (BF16 bit patterns, FP32). It holds none of the method's
arithmetic: no convolution, no normalisation, no state update. Both the CPU
oracle (test infrastructure) and the CUDA path take their inputs from here, so
the two always see bit-identical data.

Distributions follow the GLM-5.3-Flash decode workload described on the source
pages (64 heads x 128 x 128 state, kernel-4 short convolution):

* pre-conv q, k, v ~ N(0, 1), rounded to BF16 (round to nearest even);
* conv weights ~ N(0, 0.5^2) in FP32, layout [3, D, 4] (tap 3 = current token);
* conv cache ~ N(0, 1) rounded to BF16, layout [M, 3, 3, D] (tap 0 = oldest);
* beta = sigmoid(N(0, 1)) per head, FP32;
* alpha = sigmoid(N(2, 1)) per key channel, FP32 (linear-space decay);
* initial state S0 ~ N(0, 0.1^2), rounded to BF16 and widened to FP32, so that
  FP32 and BF16 state storage start from identical values.

Large normal arrays are drawn directly in float32 (numpy's float32 path);
the small per-head beta and alpha draws are float64 then stored as FP32.

Draw order for a decode layer: conv_w, conv cache, S0, then per step
(x, beta_raw, alpha_raw).  Draw order for a prefill problem: S0, q, k, v,
beta_raw, alpha_raw.  The generator is numpy's PCG64 (``default_rng``).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits",
    "bf16_widen",
    "decode_layer",
    "prefill_problem",
    "layer_seed",
    "SEED_DECODE_M1_T16",
    "SEED_DECODE_M8",
    "SEED_DECODE_M32_BF16",
    "SEED_DECODE_STACK",
    "SEED_PREFILL_M4_T4096",
    "SEED_DECODE_TOKENS",
    "gate_norm_inputs",
    "stack_tokens",
    "prefill_layer_problem",
]


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 array -> BF16 bit patterns (uint16), round to nearest even.

    Inputs here are finite normal draws, so no NaN handling is needed.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = b >> np.uint32(16)
    r &= np.uint32(1)
    r += np.uint32(0x7FFF)
    r += b
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_widen(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> the exactly equal FP32 values."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _sigmoid32(z: np.ndarray) -> np.ndarray:
    # input-distribution shaping only (beta and alpha are drawn as sigmoid of
    # a normal); evaluated in float64 and stored as FP32
    return (1.0 / (1.0 + np.exp(-z))).astype(np.float32)


# Seed spaces, 1000 seeds each, one per synthetic workload:
SEED_DECODE_M1_T16 = 0      # one layer, M = 1, 16 consecutive FP32-state steps
SEED_DECODE_M8 = 1          # one layer, M = 8, one FP32-state step
SEED_DECODE_M32_BF16 = 2    # one layer, M = 32, one BF16-state step
SEED_DECODE_STACK = 3       # the 34-layer decode stack (seed = layer index)
SEED_PREFILL_M4_T4096 = 4   # prefill, M = 4 streams x T = 4096 tokens
SEED_DECODE_TOKENS = 5      # multi-token decode (seed = token count)


def layer_seed(space: int, layer: int) -> int:
    """Per-layer seed: 1000 * space + layer, space one of the SEED_* above."""
    return 1000 * space + layer


def decode_layer(seed: int, M: int, H: int = 64, d: int = 128, T: int = 1,
                 alpha_mean: float = 2.0) -> dict:
    """Inputs for T consecutive decode steps of one KDA layer.

    Returns a dict with
      conv_w      float32 [3, D, 4]
      cache_bits  uint16  [M, 3, 3, D]   (BF16)   cache_f32: widened copy
      S0          float32 [M, H, d, d]   (BF16-representable values)
      x_bits      list of T uint16 [M, 3, D]      x_f32: widened copies
      beta        list of T float32 [M, H]
      alpha       list of T float32 [M, H, d]
    with D = H * d.
    """
    rng = np.random.default_rng(seed)
    D = H * d
    conv_w = rng.standard_normal((3, D, 4), dtype=np.float32)
    conv_w *= np.float32(0.5)
    cache_bits = bf16_bits(rng.standard_normal((M, 3, 3, D), dtype=np.float32))
    S0 = rng.standard_normal((M, H, d, d), dtype=np.float32)
    S0 *= np.float32(0.1)
    S0 = bf16_widen(bf16_bits(S0))
    x_bits, beta, alpha = [], [], []
    for _ in range(T):
        x_bits.append(bf16_bits(rng.standard_normal((M, 3, D), dtype=np.float32)))
        beta.append(_sigmoid32(rng.standard_normal((M, H))))
        alpha.append(_sigmoid32(rng.standard_normal((M, H, d)) + alpha_mean))
    return {
        "M": M, "H": H, "d": d, "T": T,
        "conv_w": conv_w,
        "cache_bits": cache_bits,
        "cache_f32": bf16_widen(cache_bits),
        "S0": np.ascontiguousarray(S0),
        "x_bits": x_bits,
        "x_f32": [bf16_widen(b) for b in x_bits],
        "beta": beta,
        "alpha": alpha,
    }


def prefill_problem(seed: int, M: int, T: int, H: int = 64, d: int = 128,
                    alpha_mean: float = 2.0) -> dict:
    """Inputs for a chunked prefill of T tokens (post-conv q, k, v).

    Returns q_bits/k_bits/v_bits uint16 [M, T, H, d] (BF16) with widened
    float32 copies q/k/v, alpha float32 [M, T, H, d], beta float32 [M, T, H]
    and S0 float32 [M, H, d, d] (BF16-representable values).
    """
    rng = np.random.default_rng(seed)
    S0 = rng.standard_normal((M, H, d, d), dtype=np.float32)
    S0 *= np.float32(0.1)
    S0 = bf16_widen(bf16_bits(S0))
    out = {"M": M, "T": T, "H": H, "d": d, "S0": np.ascontiguousarray(S0)}
    for name in ("q", "k", "v"):
        bits = bf16_bits(rng.standard_normal((M, T, H, d), dtype=np.float32))
        out[name + "_bits"] = bits
        out[name] = bf16_widen(bits)
    out["beta"] = _sigmoid32(rng.standard_normal((M, T, H)))
    out["alpha"] = _sigmoid32(rng.standard_normal((M, T, H, d), dtype=np.float32) + alpha_mean)
    return out


def gate_norm_inputs(seed: int, M: int, H: int = 64, d: int = 128, T: int = 1) -> dict:
    """Inputs of the steps fused around the decode step: the forget gate's raw
    input f ~ N(0, 1) [M, H, d] per step, A_log ~ U(-1, 1) [H], dt_bias ~
    N(0, 1) [H*d]; the output gate's input ~ N(0, 1) [M, H, d] per step and
    the RMSNorm weight ~ N(1, 0.1^2) [d]. All FP32. Draw order: A_log,
    dt_bias, norm_w, then per step (f, out_gate)."""
    rng = np.random.default_rng(seed)
    A_log = rng.uniform(-1.0, 1.0, H).astype(np.float32)
    dt_bias = rng.standard_normal(H * d).astype(np.float32)
    norm_w = (1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    f, og = [], []
    for _ in range(T):
        f.append(rng.standard_normal((M, H, d)).astype(np.float32))
        og.append(rng.standard_normal((M, H, d)).astype(np.float32))
    return {"A_log": A_log, "dt_bias": dt_bias, "norm_w": norm_w, "f": f, "out_gate": og}


def stack_tokens(layer: dict) -> dict:
    """The T steps of a ``decode_layer`` dict as token-major arrays for a
    multi-token call: x_bits uint16 [M, T, 3, D] (x_f32 widened), alpha
    float32 [M, T, H, d], beta float32 [M, T, H]."""
    x_bits = np.ascontiguousarray(np.stack(layer["x_bits"], axis=1))
    return {
        "x_bits": x_bits,
        "x_f32": bf16_widen(x_bits),
        "alpha": np.ascontiguousarray(np.stack(layer["alpha"], axis=1)),
        "beta": np.ascontiguousarray(np.stack(layer["beta"], axis=1)),
    }


def prefill_layer_problem(seed: int, M: int, T: int, H: int = 64, d: int = 128) -> dict:
    """Inputs of a KDA layer over a prompt of T tokens: pre-conv x ~ N(0, 1)
    [M, T, 3, D] and conv cache ~ N(0, 1) [M, 3, 3, D] as BF16 bits (x_bits,
    cache_bits; widened x_f32, cache_f32), conv_w ~ N(0, 0.5^2) [3, D, 4],
    the raw gate input f ~ N(0, 1) [M, T, H, d], A_log ~ U(-1, 1) [H],
    dt_bias ~ N(0, 1) [H*d], beta = sigmoid(N(0, 1)) [M, T, H], S0 ~
    N(0, 0.1^2) rounded to BF16 [M, H, d, d], the output gate ~ N(0, 1)
    [M, T, H, d] and the RMSNorm weight ~ N(1, 0.1^2) [d]. Draw order as
    listed."""
    rng = np.random.default_rng(seed)
    D = H * d
    x_bits = bf16_bits(rng.standard_normal((M, T, 3, D), dtype=np.float32))
    cache_bits = bf16_bits(rng.standard_normal((M, 3, 3, D), dtype=np.float32))
    conv_w = rng.standard_normal((3, D, 4), dtype=np.float32)
    conv_w *= np.float32(0.5)
    f = rng.standard_normal((M, T, H, d), dtype=np.float32)
    A_log = rng.uniform(-1.0, 1.0, H).astype(np.float32)
    dt_bias = rng.standard_normal(H * d).astype(np.float32)
    beta = _sigmoid32(rng.standard_normal((M, T, H)))
    S0 = rng.standard_normal((M, H, d, d), dtype=np.float32)
    S0 *= np.float32(0.1)
    S0 = bf16_widen(bf16_bits(S0))
    out_gate = rng.standard_normal((M, T, H, d), dtype=np.float32)
    norm_w = (1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    return {"M": M, "T": T, "H": H, "d": d,
            "x_bits": x_bits, "x_f32": bf16_widen(x_bits),
            "cache_bits": cache_bits, "cache_f32": bf16_widen(cache_bits),
            "conv_w": conv_w, "f": f, "A_log": A_log, "dt_bias": dt_bias, "beta": beta,
            "S0": np.ascontiguousarray(S0), "out_gate": out_gate, "norm_w": norm_w}
