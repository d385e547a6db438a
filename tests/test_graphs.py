"""Entry points captured in a CUDA graph and replayed give, bit for bit, the
results of the same call launched directly (outputs, state and conv cache).

The decode step under a graph is covered by the 34-layer stack test in
test_decode.py; these cover the other entry points. Each is called once
directly before the capture (as one warms up before capturing), then the
capture runs on fresh copies of the in-place buffers and is replayed once.
"""
import numpy as np
import pytest

from linear_attention_decode_step_gb300 import inputs
from tests.kda_testlib import bits_to_torch_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from linear_attention_decode_step_gb300 import build
    build.build()
    from linear_attention_decode_step_gb300 import kda
    return kda


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _graph_equals_direct(K, run, fresh):
    """run(bufs) launches one call on the current stream and returns the
    tensors to compare; fresh() returns new copies of the in-place buffers."""
    direct = [t.clone() for t in run(fresh())]
    torch.cuda.synchronize()
    assert K.kda_device_error() == K.KDA_OK
    bufs = fresh()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = run(bufs)
    g.replay()
    torch.cuda.synchronize()
    assert K.kda_device_error() == K.KDA_OK
    for a, b in zip(outs, direct):
        assert torch.equal(a, b)


def test_fused_decode_in_graph(K):
    M, H = 4, 16
    inp = inputs.decode_layer(9700, M=M, H=H, T=1)
    gn = inputs.gate_norm_inputs(9701, M=M, H=H, T=1)
    x = bits_to_torch_bf16(inp["x_bits"][0], "cuda")
    w, f, A, b = _dev(inp["conv_w"]), _dev(gn["f"][0]), _dev(gn["A_log"]), _dev(gn["dt_bias"])
    beta, og, nw = _dev(inp["beta"][0]), _dev(gn["out_gate"][0]), _dev(gn["norm_w"])

    def fresh():
        return (bits_to_torch_bf16(inp["cache_bits"], "cuda"), _dev(inp["S0"]),
                torch.empty((M, H, 128), dtype=torch.float32, device="cuda"))

    def run(bufs):
        cache, S, y = bufs
        K.kda_decode_step_fused(x, w, cache, f, A, b, beta, S, y, out_gate=og, norm_weight=nw)
        return y, S, cache

    _graph_equals_direct(K, run, fresh)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_tokens_in_graph(K, state_dtype):
    M, H, T = 4, 16, 4
    inp = inputs.decode_layer(9800, M=M, H=H, T=T)
    tok = inputs.stack_tokens(inp)
    x, w = bits_to_torch_bf16(tok["x_bits"], "cuda"), _dev(inp["conv_w"])
    alpha, beta = _dev(tok["alpha"]), _dev(tok["beta"])

    def fresh():
        S = _dev(inp["S0"])
        return (bits_to_torch_bf16(inp["cache_bits"], "cuda"),
                S.to(torch.bfloat16) if state_dtype == "bf16" else S,
                torch.empty((M, T, H, 128), dtype=torch.float32, device="cuda"))

    def run(bufs):
        cache, S, o = bufs
        K.kda_decode_tokens(x, w, cache, alpha, beta, S, o)
        return o, S, cache

    _graph_equals_direct(K, run, fresh)


@pytest.mark.parametrize("kernel", [1, 2])  # KDA_PREFILL_SIMT, KDA_PREFILL_TC
def test_chunk_prefill_in_graph(K, kernel):
    M, T, H = 2, 130, 4
    p = inputs.prefill_problem(9900, M=M, T=T, H=H)
    q, k, v = (bits_to_torch_bf16(p[n + "_bits"], "cuda") for n in ("q", "k", "v"))
    alpha, beta = _dev(p["alpha"]), _dev(p["beta"])

    def fresh():
        return _dev(p["S0"]), torch.empty((M, T, H, 128), dtype=torch.float32, device="cuda")

    def run(bufs):
        S, o = bufs
        K.kda_chunk_prefill_config(q, k, v, alpha, beta, S, o, kernel=kernel)
        return o, S

    _graph_equals_direct(K, run, fresh)


def test_prefill_layer_in_graph(K):
    M, T, H = 2, 130, 4
    p = inputs.prefill_layer_problem(9950, M=M, T=T, H=H)
    x, w = bits_to_torch_bf16(p["x_bits"], "cuda"), _dev(p["conv_w"])
    f, A, b, beta = _dev(p["f"]), _dev(p["A_log"]), _dev(p["dt_bias"]), _dev(p["beta"])
    og, nw = _dev(p["out_gate"]), _dev(p["norm_w"])

    def fresh():
        return (bits_to_torch_bf16(p["cache_bits"], "cuda"), _dev(p["S0"]),
                torch.empty((M, T, H, 128), dtype=torch.float32, device="cuda"))

    def run(bufs):
        cache, S, y = bufs
        K.kda_prefill_layer(x, w, cache, f, A, b, beta, S, y, out_gate=og, norm_weight=nw)
        return y, S, cache

    _graph_equals_direct(K, run, fresh)
