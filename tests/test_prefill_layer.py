"""GPU parity of the KDA layer over a prompt (kda_prefill_layer: conv + SiLU
with the cache as left context, forget gate, chunked recurrence on the tensor
cores, optional gated RMSNorm) against the fp64 oracle's prefill_layer (the
gate, then T decode steps, then the norm): max |gpu - oracle| / max |oracle|
<= 5e-3 on every output and on the final state; the conv cache bit-exact."""
import numpy as np
import pytest

import oracle
from linear_attention_decode_step_gb300 import inputs
from tests.kda_testlib import (bits_to_torch_bf16, oracle_prefill_layer_all_heads, rel_err,
                               rel_err_per_head, to_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = 5e-3


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from linear_attention_decode_step_gb300 import build
    build.build()
    from linear_attention_decode_step_gb300 import kda
    return kda


def _run(K, p, x_dtype="bf16", norm=True, scale=1.0):
    dev = "cuda"
    if x_dtype == "bf16":
        x = bits_to_torch_bf16(p["x_bits"], dev)
        cache = bits_to_torch_bf16(p["cache_bits"], dev)
    else:
        x = torch.from_numpy(p["x_f32"]).to(dev)
        cache = torch.from_numpy(p["cache_f32"]).to(dev)
    t = lambda n: torch.from_numpy(p[n]).to(dev)
    S = t("S0").clone()
    y = K.kda_prefill_layer(x, t("conv_w"), cache, t("f"), t("A_log"), t("dt_bias"), t("beta"), S,
                            scale=scale, out_gate=t("out_gate") if norm else None,
                            norm_weight=t("norm_w") if norm else None)
    torch.cuda.synchronize()
    assert K.kda_device_error() == K.KDA_OK
    return y.double().cpu().numpy(), S.double().cpu().numpy(), to_f64(cache)


def _oracle(p, norm=True, scale=1.0, sl=None):
    g = (lambda a: a) if sl is None else (lambda a: a[sl])
    return oracle.prefill_layer(g(p["x_f32"]), p["conv_w"], g(p["cache_f32"]), g(p["f"]),
                                p["A_log"], p["dt_bias"], g(p["beta"]), g(p["S0"]), scale=scale,
                                out_gate=g(p["out_gate"]) if norm else None,
                                norm_w=p["norm_w"] if norm else None)


@pytest.mark.parametrize("T", [1, 2, 3, 17, 64, 65, 130])
def test_layer_lengths(K, T):
    p = inputs.prefill_layer_problem(6000 + T, M=2, T=T, H=3)
    y, S, c = _run(K, p)
    y_ref, S_ref, c_ref = _oracle(p)
    assert rel_err(y, y_ref) <= TOL, rel_err(y, y_ref)
    assert rel_err(S, S_ref) <= TOL, rel_err(S, S_ref)
    np.testing.assert_array_equal(c, c_ref)


@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_layer_without_norm_and_scaled(K, x_dtype):
    p = inputs.prefill_layer_problem(6100, M=1, T=100, H=2)
    y, S, c = _run(K, p, x_dtype=x_dtype, norm=False, scale=128 ** -0.5)
    y_ref, S_ref, c_ref = _oracle(p, norm=False, scale=128 ** -0.5)
    assert rel_err(y, y_ref) <= TOL
    assert rel_err(S, S_ref) <= TOL
    np.testing.assert_array_equal(c, c_ref)


def test_layer_zero_input_only_decays(K):
    """All-zero pre-conv inputs and cache: q = k = v = 0 after the conv, so
    every output (after the gated norm too) is exactly 0, the state is only
    faded by the gate's decay, and the cache stays zero."""
    p = inputs.prefill_layer_problem(6300, M=2, T=100, H=3)
    for n in ("x_bits", "x_f32", "cache_bits", "cache_f32"):
        p[n] = np.zeros_like(p[n])
    y, S, c = _run(K, p)
    assert np.all(y == 0.0)
    y_ref, S_ref, c_ref = _oracle(p)
    assert rel_err(S, S_ref) <= TOL
    np.testing.assert_array_equal(c, c_ref)


def test_layer_matches_decode_steps_on_device(K):
    """Prefill of 9 tokens equals 9 fused decode steps on the GPU (same
    inputs, state and cache carried)."""
    p = inputs.prefill_layer_problem(6200, M=2, T=9, H=4)
    y, S, c = _run(K, p)
    dev = "cuda"
    x = bits_to_torch_bf16(p["x_bits"], dev)
    cache = bits_to_torch_bf16(p["cache_bits"], dev)
    t = lambda n: torch.from_numpy(p[n]).to(dev)
    S2 = t("S0").clone()
    for k in range(9):
        yk = K.kda_decode_step_fused(x[:, k].contiguous(), t("conv_w"), cache,
                                     t("f")[:, k].contiguous(), t("A_log"), t("dt_bias"),
                                     t("beta")[:, k].contiguous(), S2,
                                     out_gate=t("out_gate")[:, k].contiguous(),
                                     norm_weight=t("norm_w"))
        assert rel_err(y[:, k], yk.double().cpu().numpy()) <= TOL
    torch.cuda.synchronize()
    assert rel_err(S, S2.double().cpu().numpy()) <= TOL
    np.testing.assert_array_equal(c, to_f64(cache))


def test_layer_M4_T4096_every_head(K):
    """M=4 streams, T=4096 tokens, 64 heads (the prefill workload) as a whole
    layer with the gated norm: every output and the final state of all 256
    (stream, head) pairs against 4096 oracle steps each (oracle on all host
    cores), each pair to the bar on its own; the conv cache bit for bit."""
    p = inputs.prefill_layer_problem(inputs.layer_seed(inputs.SEED_PREFILL_M4_T4096, 1), M=4, T=4096, H=64)
    y, S, c = _run(K, p)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(S))
    y_ref, S_ref, c_ref = oracle_prefill_layer_all_heads(p)
    ey = rel_err_per_head(y, y_ref, (0, 2))
    eS = rel_err_per_head(S, S_ref, (0, 1))
    assert float(ey.max()) <= TOL, ("y", np.unravel_index(ey.argmax(), ey.shape), float(ey.max()))
    assert float(eS.max()) <= TOL, ("S", np.unravel_index(eS.argmax(), eS.shape), float(eS.max()))
    np.testing.assert_array_equal(c, c_ref)


@pytest.mark.parametrize("M,T,H", [(1, 70, 1), (3, 129, 5)])
def test_layer_odd_shapes(K, M, T, H):
    """One head, and an odd head count with a ragged third chunk, through the
    5-D tensor maps over x [M][T][3][H*128]."""
    p = inputs.prefill_layer_problem(6300 + H, M=M, T=T, H=H)
    y, S, c = _run(K, p)
    y_ref, S_ref, c_ref = _oracle(p)
    assert rel_err(y, y_ref) <= TOL, rel_err(y, y_ref)
    assert rel_err(S, S_ref) <= TOL, rel_err(S, S_ref)
    np.testing.assert_array_equal(c, c_ref)


def test_layer_pieces_equal_whole_sequences(K):
    """The layer form at M = 3 x 64 heads x 1000 tokens (pieces in rounds, as
    in test_prefill.py): each stream equals a call of that stream alone bit for
    bit, outputs, final state and conv cache (a later piece takes its conv
    window from x, the first from the cache; only the last writes the cache)."""
    p = inputs.prefill_layer_problem(8710, M=3, T=1000, H=64)
    y, S, cache = _run(K, p)
    for m in range(3):
        per_stream = ("x_bits", "x_f32", "cache_bits", "cache_f32", "f", "beta", "S0", "out_gate")
        one = {n: (v[m:m + 1].copy() if n in per_stream else v) for n, v in p.items()}
        y1, S1, c1 = _run(K, one)
        np.testing.assert_array_equal(y1[0], y[m])
        np.testing.assert_array_equal(S1[0], S[m])
        np.testing.assert_array_equal(c1[0], cache[m])
