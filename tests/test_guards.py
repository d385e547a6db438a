"""Guard regions around every device buffer of every entry point.

Each input and output of a call sits between two 4 KiB guard regions filled
with a known byte. After the call, on small and ragged shapes (odd head
counts, prompts that end inside a chunk), the checks are:

* no guard byte changed: nothing is written just before or after a buffer;
* read-only inputs are bit-for-bit unchanged;
* every element of an output was written: outputs start as all-ones bytes
  (a NaN in FP32) and none may remain;
* the results still match the fp64 oracle at the usual bars, so the guarded
  run did the real work.

These checks stand in for a memory checker, which this test setup cannot
run. They catch writes past a buffer's edges and outputs left unwritten.
"""
import numpy as np
import pytest

import oracle
from linear_attention_decode_step_gb300 import inputs
from tests.kda_testlib import (TOL_BF16_STATE, TOL_F32_STATE, bits_to_torch_bf16, rel_err,
                               to_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GUARD = 4096        # bytes on each side; keeps the buffer itself 16-byte aligned
GUARD_BYTE = 0xA5
OUT_BYTE = 0xFF     # an FP32 (and BF16) NaN pattern for outputs not yet written
TOL_PREFILL = 5e-3


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from linear_attention_decode_step_gb300 import build
    build.build()
    from linear_attention_decode_step_gb300 import kda
    return kda


class Guarded:
    """Device buffers, each between two guard regions of GUARD_BYTE."""

    def __init__(self):
        self.bufs = []

    def _alloc(self, name, shape, dtype, fill):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((2 * GUARD + n,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
        raw[GUARD:GUARD + n] = fill
        view = raw[GUARD:GUARD + n].view(dtype).view(shape)
        assert view.data_ptr() % 16 == 0
        return raw, n, view

    def input(self, name, t):
        """A read-only input: a guarded copy of t."""
        raw, n, view = self._alloc(name, tuple(t.shape), t.dtype, 0)
        view.copy_(t)
        self.bufs.append((name, raw, n, view, view.clone(), False))
        return view

    def inout(self, name, t):
        """A buffer updated in place: a guarded copy of t."""
        raw, n, view = self._alloc(name, tuple(t.shape), t.dtype, 0)
        view.copy_(t)
        self.bufs.append((name, raw, n, view, None, False))
        return view

    def output(self, name, shape, dtype=torch.float32):
        """An output: guarded, every byte OUT_BYTE until the call writes it."""
        raw, n, view = self._alloc(name, shape, dtype, OUT_BYTE)
        self.bufs.append((name, raw, n, view, None, True))
        return view

    def check(self):
        torch.cuda.synchronize()
        for name, raw, n, view, snap, is_out in self.bufs:
            assert bool((raw[:GUARD] == GUARD_BYTE).all()), "%s: guard before it written" % name
            assert bool((raw[GUARD + n:] == GUARD_BYTE).all()), "%s: guard after it written" % name
            if snap is not None:
                assert torch.equal(view, snap), "%s: read-only input modified" % name
            if is_out:
                assert not bool(torch.isnan(view.float()).any()), "%s: elements not written" % name


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _x(inp, key_bits, key_f32, x_dtype):
    return bits_to_torch_bf16(inp[key_bits], "cuda") if x_dtype == "bf16" else _dev(inp[key_f32])


def _state(S0, state_dtype):
    S = _dev(S0)
    return S.to(torch.bfloat16) if state_dtype == "bf16" else S


def _tol(state_dtype):
    return TOL_BF16_STATE if state_dtype == "bf16" else TOL_F32_STATE


@pytest.mark.parametrize("kernel,tile", [("auto", None), ("stream", None),
                                         ("cluster", (32, 128)), ("cluster", (16, 64))])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_decode_step_guards(K, kernel, tile, state_dtype, x_dtype):
    M, H = 3, 5
    inp = inputs.decode_layer(9100, M=M, H=H, T=1)
    g = Guarded()
    x = g.input("x", bits_to_torch_bf16(inp["x_bits"][0], "cuda") if x_dtype == "bf16"
                else _dev(inp["x_f32"][0]))
    w = g.input("conv_w", _dev(inp["conv_w"]))
    cache = g.inout("conv_cache", _x(inp, "cache_bits", "cache_f32", x_dtype))
    alpha = g.input("alpha", _dev(inp["alpha"][0]))
    beta = g.input("beta", _dev(inp["beta"][0]))
    S = g.inout("state", _state(inp["S0"], state_dtype))
    o = g.output("o", (M, H, 128))
    if kernel == "auto":
        K.kda_decode_step(x, w, cache, alpha, beta, S, o)
    elif kernel == "stream":
        K.kda_decode_step_config(x, w, cache, alpha, beta, S, o, kernel=K.KDA_DECODE_STREAM)
    else:
        K.kda_decode_step_config(x, w, cache, alpha, beta, S, o, kernel=K.KDA_DECODE_CLUSTER,
                                 columns=tile[0], threads=tile[1])
    g.check()
    assert K.kda_device_error() == K.KDA_OK
    o_ref, S_ref, c_ref = oracle.decode_step(inp["x_f32"][0], inp["conv_w"], inp["cache_f32"],
                                             inp["alpha"][0], inp["beta"][0], inp["S0"])
    assert rel_err(o.double().cpu().numpy(), o_ref) <= _tol(state_dtype)
    assert rel_err(to_f64(S), S_ref) <= _tol(state_dtype)
    np.testing.assert_array_equal(to_f64(cache), c_ref)


@pytest.mark.parametrize("norm", [True, False])
def test_decode_step_fused_guards(K, norm):
    M, H = 3, 5
    inp = inputs.decode_layer(9200, M=M, H=H, T=1)
    gn = inputs.gate_norm_inputs(9201, M=M, H=H, T=1)
    g = Guarded()
    x = g.input("x", bits_to_torch_bf16(inp["x_bits"][0], "cuda"))
    w = g.input("conv_w", _dev(inp["conv_w"]))
    cache = g.inout("conv_cache", bits_to_torch_bf16(inp["cache_bits"], "cuda"))
    f = g.input("gate_f", _dev(gn["f"][0]))
    A = g.input("A_log", _dev(gn["A_log"]))
    b = g.input("dt_bias", _dev(gn["dt_bias"]))
    beta = g.input("beta", _dev(inp["beta"][0]))
    S = g.inout("state", _state(inp["S0"], "f32"))
    og = g.input("out_gate", _dev(gn["out_gate"][0])) if norm else None
    nw = g.input("norm_w", _dev(gn["norm_w"])) if norm else None
    y = g.output("y", (M, H, 128))
    K.kda_decode_step_fused(x, w, cache, f, A, b, beta, S, y, out_gate=og, norm_weight=nw)
    g.check()
    assert K.kda_device_error() == K.KDA_OK
    y_ref, S_ref, c_ref = oracle.decode_step_fused(
        inp["x_f32"][0], inp["conv_w"], inp["cache_f32"], gn["f"][0], gn["A_log"],
        gn["dt_bias"], inp["beta"][0], inp["S0"],
        out_gate=gn["out_gate"][0] if norm else None, norm_w=gn["norm_w"] if norm else None)
    assert rel_err(y.double().cpu().numpy(), y_ref) <= TOL_F32_STATE
    assert rel_err(to_f64(S), S_ref) <= TOL_F32_STATE
    np.testing.assert_array_equal(to_f64(cache), c_ref)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_tokens_guards(K, state_dtype):
    M, H, T = 3, 5, 5
    inp = inputs.decode_layer(9300, M=M, H=H, T=T)
    tok = inputs.stack_tokens(inp)
    g = Guarded()
    x = g.input("x", bits_to_torch_bf16(tok["x_bits"], "cuda"))
    w = g.input("conv_w", _dev(inp["conv_w"]))
    cache = g.inout("conv_cache", bits_to_torch_bf16(inp["cache_bits"], "cuda"))
    alpha = g.input("alpha", _dev(tok["alpha"]))
    beta = g.input("beta", _dev(tok["beta"]))
    S = g.inout("state", _state(inp["S0"], state_dtype))
    o = g.output("o", (M, T, H, 128))
    K.kda_decode_tokens(x, w, cache, alpha, beta, S, o)
    g.check()
    assert K.kda_device_error() == K.KDA_OK
    o_ref, S_ref, c_ref = oracle.decode_tokens(tok["x_f32"], inp["conv_w"], inp["cache_f32"],
                                               tok["alpha"], tok["beta"], inp["S0"])
    assert rel_err(o.double().cpu().numpy(), o_ref) <= _tol(state_dtype)
    assert rel_err(to_f64(S), S_ref) <= _tol(state_dtype)
    np.testing.assert_array_equal(to_f64(cache), c_ref)


@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_conv_step_guards(K, x_dtype):
    M, H = 3, 5
    D = H * 128
    inp = inputs.decode_layer(9400, M=M, H=H, T=1)
    g = Guarded()
    x = g.input("x", bits_to_torch_bf16(inp["x_bits"][0], "cuda") if x_dtype == "bf16"
                else _dev(inp["x_f32"][0]))
    w = g.input("conv_w", _dev(inp["conv_w"]))
    cache = g.inout("conv_cache", _x(inp, "cache_bits", "cache_f32", x_dtype))
    y = g.output("y", (M, 3, D))
    K.kda_conv_step(x, w, cache, y)
    g.check()
    y_ref, c_ref = oracle.conv_step(inp["x_f32"][0], inp["conv_w"], inp["cache_f32"])
    assert rel_err(y.double().cpu().numpy(), y_ref) <= 1e-5
    np.testing.assert_array_equal(to_f64(cache), c_ref)


@pytest.mark.parametrize("kernel", [1, 2])  # KDA_PREFILL_SIMT, KDA_PREFILL_TC
@pytest.mark.parametrize("qkv", ["bf16", "f32"])
def test_chunk_prefill_guards(K, kernel, qkv):
    M, T, H = 2, 70, 3
    p = inputs.prefill_problem(9500, M=M, T=T, H=H)
    g = Guarded()
    q, k, v = (g.input(n, bits_to_torch_bf16(p[n + "_bits"], "cuda") if qkv == "bf16"
                       else _dev(p[n])) for n in ("q", "k", "v"))
    alpha = g.input("alpha", _dev(p["alpha"]))
    beta = g.input("beta", _dev(p["beta"]))
    S = g.inout("state", _dev(p["S0"]))
    o = g.output("o", (M, T, H, 128))
    K.kda_chunk_prefill_config(q, k, v, alpha, beta, S, o, kernel=kernel)
    g.check()
    assert K.kda_device_error() == K.KDA_OK
    o_ref, S_ref = oracle.recurrent(p["q"], p["k"], p["v"], p["alpha"], p["beta"], p["S0"])
    assert rel_err(o.double().cpu().numpy(), o_ref) <= TOL_PREFILL
    assert rel_err(S.double().cpu().numpy(), S_ref) <= TOL_PREFILL


@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("norm", [True, False])
def test_prefill_layer_guards(K, x_dtype, norm):
    M, T, H = 2, 70, 3
    p = inputs.prefill_layer_problem(9600, M=M, T=T, H=H)
    g = Guarded()
    x = g.input("x", _x(p, "x_bits", "x_f32", x_dtype))
    w = g.input("conv_w", _dev(p["conv_w"]))
    cache = g.inout("conv_cache", _x(p, "cache_bits", "cache_f32", x_dtype))
    f = g.input("gate_f", _dev(p["f"]))
    A = g.input("A_log", _dev(p["A_log"]))
    b = g.input("dt_bias", _dev(p["dt_bias"]))
    beta = g.input("beta", _dev(p["beta"]))
    S = g.inout("state", _dev(p["S0"]))
    og = g.input("out_gate", _dev(p["out_gate"])) if norm else None
    nw = g.input("norm_w", _dev(p["norm_w"])) if norm else None
    y = g.output("y", (M, T, H, 128))
    K.kda_prefill_layer(x, w, cache, f, A, b, beta, S, y, out_gate=og, norm_weight=nw)
    g.check()
    assert K.kda_device_error() == K.KDA_OK
    y_ref, S_ref, c_ref = oracle.prefill_layer(
        p["x_f32"], p["conv_w"], p["cache_f32"], p["f"], p["A_log"], p["dt_bias"], p["beta"],
        p["S0"], out_gate=p["out_gate"] if norm else None, norm_w=p["norm_w"] if norm else None)
    assert rel_err(y.double().cpu().numpy(), y_ref) <= TOL_PREFILL
    assert rel_err(S.double().cpu().numpy(), S_ref) <= TOL_PREFILL
    np.testing.assert_array_equal(to_f64(cache), c_ref)
