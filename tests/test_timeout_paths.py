"""The library's own kernels leave through their timeout path and report it.

Every device-side wait of the streaming decode, the multi-token decode and
the tensor-core prefill is bounded. A second build of those three kernels'
sources with a zero wait budget, polling instead of suspending
(-DKDA_WAIT_BUDGET=0 -DKDA_WAIT_POLL), makes their first waits give up
before the bulk and tensor copies they wait for have landed: valid inputs,
ordinary buffers and tensor maps, no fault. Each call through that build's
C ABI must then
  * return normally, with kda_device_error() = KDA_ERR_TIMEOUT (every thread
    of the group or CTA leaves together, the copies and tensor-core products
    in flight land before the shared and tensor memory are released, the
    tensor memory is freed);
  * leave the context usable: the same call through the regular library
    right after is correct against the oracle and reports KDA_OK.
"""
import ctypes

import numpy as np
import pytest

import oracle
from linear_attention_decode_step_gb300 import inputs
from tests.kda_testlib import DeviceLayer, bits_to_torch_bf16, oracle_layer, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SHORT_WAIT_SOURCES = ["kda_decode_stream.cu", "kda_decode_tokens.cu", "kda_prefill_tc.cu"]


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from linear_attention_decode_step_gb300 import build, kda
    path = build.build_variant("shortwait", ["KDA_WAIT_BUDGET=0", "KDA_WAIT_POLL"],
                               SHORT_WAIT_SOURCES)
    short = kda.load(path)
    assert short.kda_device_error(None) == kda.KDA_OK  # its own, fresh error words
    return kda, short


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_step_times_out_then_library_is_usable(libs, state_dtype):
    kda, short = libs
    inp = inputs.decode_layer(8100, M=8, T=1)
    dl = DeviceLayer(inp, state_dtype)
    sd = kda.KDA_BF16 if state_dtype == "bf16" else kda.KDA_F32
    st = short.kda_decode_step(_p(dl.x[0]), kda.KDA_BF16, _p(dl.conv_w), _p(dl.cache), kda.KDA_BF16,
                               _p(dl.alpha[0]), _p(dl.beta[0]), _p(dl.state), sd, 1.0, _p(dl.o),
                               8, 64, 128, 128, None)
    assert st == kda.KDA_OK
    assert short.kda_device_error(None) == kda.KDA_ERR_TIMEOUT
    assert short.kda_device_error(None) == kda.KDA_OK  # read and cleared
    # the regular build on fresh buffers
    dl = DeviceLayer(inp, state_dtype)
    kda.kda_decode_step(dl.x[0], dl.conv_w, dl.cache, dl.alpha[0], dl.beta[0], dl.state, dl.o)
    torch.cuda.synchronize()
    assert kda.kda_device_error() == kda.KDA_OK
    ref, S, _ = oracle_layer(inp)
    tol = 5e-3 if state_dtype == "bf16" else 1e-4
    assert rel_err(dl.o.double().cpu().numpy(), ref[0]) <= tol


@pytest.mark.parametrize("T", [2, 4, 12])
def test_decode_tokens_times_out_then_library_is_usable(libs, T):
    """T = 2 runs the token-by-token kernel, 4 the chunked kernel with one
    chunk, 12 the chunked kernel with two."""
    kda, short = libs
    inp = inputs.decode_layer(8200, M=8, T=T)
    tok = inputs.stack_tokens(inp)
    dev = "cuda"

    def bufs():
        return (bits_to_torch_bf16(tok["x_bits"], dev), torch.from_numpy(inp["conv_w"]).to(dev),
                bits_to_torch_bf16(inp["cache_bits"], dev), torch.from_numpy(tok["alpha"]).to(dev),
                torch.from_numpy(tok["beta"]).to(dev), torch.from_numpy(inp["S0"]).to(dev).clone(),
                torch.empty((8, T, 64, 128), dtype=torch.float32, device=dev))
    x, w, cache, alpha, beta, S, o = bufs()
    st = short.kda_decode_tokens(_p(x), kda.KDA_BF16, _p(w), _p(cache), kda.KDA_BF16, _p(alpha),
                                 _p(beta), _p(S), kda.KDA_F32, 1.0, _p(o), 8, T, 64, 128, 128, None)
    assert st == kda.KDA_OK
    assert short.kda_device_error(None) == kda.KDA_ERR_TIMEOUT
    x, w, cache, alpha, beta, S, o = bufs()
    kda.kda_decode_tokens(x, w, cache, alpha, beta, S, o)
    torch.cuda.synchronize()
    assert kda.kda_device_error() == kda.KDA_OK
    o_ref, S_ref, _ = oracle.decode_tokens(tok["x_f32"], inp["conv_w"], inp["cache_f32"],
                                           tok["alpha"], tok["beta"], inp["S0"])
    assert rel_err(o.double().cpu().numpy(), o_ref) <= 1e-4
    assert rel_err(S.double().cpu().numpy(), S_ref) <= 1e-4


def test_chunk_prefill_times_out_then_library_is_usable(libs):
    kda, short = libs
    p = inputs.prefill_problem(8300, M=2, T=200, H=8)
    dev = "cuda"

    def bufs():
        q, k, v = (bits_to_torch_bf16(p[n + "_bits"], dev) for n in ("q", "k", "v"))
        return (q, k, v, torch.from_numpy(p["alpha"]).to(dev), torch.from_numpy(p["beta"]).to(dev),
                torch.from_numpy(p["S0"]).to(dev).clone(),
                torch.empty((2, 200, 8, 128), dtype=torch.float32, device=dev))
    q, k, v, alpha, beta, S, o = bufs()
    st = short.kda_chunk_prefill_config(_p(q), _p(k), _p(v), kda.KDA_BF16, _p(alpha), _p(beta),
                                        _p(S), _p(o), 1.0, 2, 200, 8, 128, 128, 64,
                                        kda.KDA_PREFILL_TC, None)
    assert st == kda.KDA_OK
    assert short.kda_device_error(None) == kda.KDA_ERR_TIMEOUT
    # twice in a row: the first call freed its tensor memory (an allocation
    # left behind would make the next one wait for columns that never free)
    st = short.kda_chunk_prefill_config(_p(q), _p(k), _p(v), kda.KDA_BF16, _p(alpha), _p(beta),
                                        _p(S), _p(o), 1.0, 2, 200, 8, 128, 128, 64,
                                        kda.KDA_PREFILL_TC, None)
    assert st == kda.KDA_OK
    assert short.kda_device_error(None) == kda.KDA_ERR_TIMEOUT
    q, k, v, alpha, beta, S, o = bufs()
    kda.kda_chunk_prefill(q, k, v, alpha, beta, S, o)
    torch.cuda.synchronize()
    assert kda.kda_device_error() == kda.KDA_OK
    o_ref, S_ref = oracle.recurrent(p["q"], p["k"], p["v"], p["alpha"], p["beta"], p["S0"])
    assert rel_err(o.double().cpu().numpy(), o_ref) <= 5e-3
    assert rel_err(S.double().cpu().numpy(), S_ref) <= 5e-3


def test_prefill_layer_times_out_then_library_is_usable(libs):
    kda, short = libs
    p = inputs.prefill_layer_problem(8400, M=1, T=130, H=4)
    dev = "cuda"
    t = lambda n: torch.from_numpy(p[n]).to(dev)

    def bufs():
        return (bits_to_torch_bf16(p["x_bits"], dev), bits_to_torch_bf16(p["cache_bits"], dev),
                t("S0").clone(), torch.empty((1, 130, 4, 128), dtype=torch.float32, device=dev))
    x, cache, S, y = bufs()
    w, f, A, b, beta, og, nw = (t(n) for n in ("conv_w", "f", "A_log", "dt_bias", "beta",
                                               "out_gate", "norm_w"))
    st = short.kda_prefill_layer(_p(x), kda.KDA_BF16, _p(w), _p(cache), kda.KDA_BF16, _p(f), _p(A),
                                 _p(b), -5.0, _p(beta), _p(S), 1.0, _p(og), _p(nw), 1e-5, _p(y),
                                 1, 130, 4, 128, 128, 64, None)
    assert st == kda.KDA_OK
    assert short.kda_device_error(None) == kda.KDA_ERR_TIMEOUT
    x, cache, S, y = bufs()
    kda.kda_prefill_layer(x, w, cache, f, A, b, beta, S, y, out_gate=og, norm_weight=nw)
    torch.cuda.synchronize()
    assert kda.kda_device_error() == kda.KDA_OK
    y_ref, S_ref, _ = oracle.prefill_layer(p["x_f32"], p["conv_w"], p["cache_f32"], p["f"],
                                           p["A_log"], p["dt_bias"], p["beta"], p["S0"],
                                           out_gate=p["out_gate"], norm_w=p["norm_w"])
    assert rel_err(y.double().cpu().numpy(), y_ref) <= 5e-3
    assert rel_err(S.double().cpu().numpy(), S_ref) <= 5e-3
