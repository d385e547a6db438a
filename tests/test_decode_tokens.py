"""GPU parity of the multi-token decode (kda_decode_tokens: T decode steps in
one launch) against the fp64 oracle's decode_tokens: 1e-4 (FP32 state) /
5e-3 (BF16 state) on every token's o and on the final state; the conv cache
bit-exact."""
import numpy as np
import pytest

import oracle
from linear_attention_decode_step_gb300 import inputs
from tests.kda_testlib import (TOL_BF16_STATE, TOL_F32_STATE, bits_to_torch_bf16, rel_err,
                               to_f64)

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


def _device(inp, tok, state_dtype, x_dtype):
    dev = "cuda"
    if x_dtype == "bf16":
        x = bits_to_torch_bf16(tok["x_bits"], dev)
        cache = bits_to_torch_bf16(inp["cache_bits"], dev)
    else:
        x = torch.from_numpy(tok["x_f32"]).to(dev)
        cache = torch.from_numpy(inp["cache_f32"]).to(dev)
    S = torch.from_numpy(inp["S0"]).to(dev)
    S = S.to(torch.bfloat16) if state_dtype == "bf16" else S.clone()
    return (x, torch.from_numpy(inp["conv_w"]).to(dev), cache,
            torch.from_numpy(tok["alpha"]).to(dev), torch.from_numpy(tok["beta"]).to(dev), S)


def _check(K, M, H, T, state_dtype="f32", x_dtype="bf16", scale=1.0, seed=0, edit=None):
    """Runs T tokens through kda_decode_tokens and checks them against the
    oracle; `edit(inp, tok)` may overwrite the drawn inputs first. Returns the
    device outputs (o, final state, initial state)."""
    inp = inputs.decode_layer(8000 + seed, M=M, H=H, T=T)
    tok = inputs.stack_tokens(inp)
    if edit is not None:
        edit(inp, tok)
    x, w, cache, alpha, beta, S = _device(inp, tok, state_dtype, x_dtype)
    S_before = S.clone()
    o = K.kda_decode_tokens(x, w, cache, alpha, beta, S, scale=scale)
    torch.cuda.synchronize()
    assert K.kda_device_error() == K.KDA_OK
    o_ref, S_ref, c_ref = oracle.decode_tokens(tok["x_f32"], inp["conv_w"], inp["cache_f32"],
                                               tok["alpha"], tok["beta"], inp["S0"], scale=scale)
    tol = TOL_BF16_STATE if state_dtype == "bf16" else TOL_F32_STATE
    o = o.double().cpu().numpy()
    for t in range(T):
        assert rel_err(o[:, t], o_ref[:, t]) <= tol, (t, rel_err(o[:, t], o_ref[:, t]))
    assert rel_err(to_f64(S), S_ref) <= tol, rel_err(to_f64(S), S_ref)
    np.testing.assert_array_equal(to_f64(cache), c_ref)
    return o, S, S_before


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 7, 8, 9, 16, 17])
def test_tokens_lengths(K, T):
    _check(K, 2, 8, T, seed=T)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_tokens_dtypes(K, state_dtype, x_dtype):
    _check(K, 3, 5, 5, state_dtype, x_dtype, scale=128 ** -0.5, seed=30)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [2, 4])
def test_tokens_M32_full_heads(K, state_dtype, T):
    """M = 32 streams x 64 heads (the decode workload), 2 tokens (token by
    token, the conv cache by a tensor copy) and 4 (chunked): every output and
    the whole final state against the oracle."""
    _check(K, 32, 64, T, state_dtype, seed=40 + T)


def test_tokens_single_stream_single_head(K):
    _check(K, 1, 1, 6, seed=50)


def test_tokens_long_run(K):
    """64 tokens in one call (the longest draft the page's MTP use suggests)."""
    _check(K, 2, 4, 64, seed=60)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_tokens_identity_leaves_state(K, state_dtype):
    """alpha = 1, beta = 0 for every token: the state comes back bit for bit
    (the fade multiplies by exactly 1, the correction adds exactly 0) and each
    o_t = S0^T q_t."""
    def identity(inp, tok):
        tok["alpha"] = np.ones_like(tok["alpha"])
        tok["beta"] = np.zeros_like(tok["beta"])
    _, S, S_before = _check(K, 3, 6, 5, state_dtype, seed=70, edit=identity)
    assert torch.equal(S, S_before)


def test_tokens_zero_input_degenerate(K):
    """All-zero pre-conv inputs and cache: q = k = v = 0 after the conv, so
    every o_t is exactly 0 and the state is only faded, token by token."""
    def zero(inp, tok):
        for n in ("x_bits", "x_f32"):
            tok[n] = np.zeros_like(tok[n])
        for n in ("cache_bits", "cache_f32"):
            inp[n] = np.zeros_like(inp[n])
    o, _, _ = _check(K, 2, 4, 6, seed=80, edit=zero)
    assert np.all(o == 0.0)


def test_one_token_matches_decode_step(K):
    """T = 1 is exactly one decode step: same outputs as kda_decode_step."""
    inp = inputs.decode_layer(8100, M=4, H=16, T=1)
    tok = inputs.stack_tokens(inp)
    x, w, cache, alpha, beta, S = _device(inp, tok, "f32", "bf16")
    x2, w2, cache2, alpha2, beta2, S2 = _device(inp, tok, "f32", "bf16")
    o = K.kda_decode_tokens(x, w, cache, alpha, beta, S)
    o2 = K.kda_decode_step(x2[:, 0].contiguous(), w2, cache2, alpha2[:, 0].contiguous(),
                           beta2[:, 0].contiguous(), S2)
    torch.cuda.synchronize()
    assert rel_err(o[:, 0].double().cpu().numpy(), o2.double().cpu().numpy()) <= 1e-6
    assert rel_err(to_f64(S), to_f64(S2)) <= 1e-6
    assert torch.equal(cache, cache2)


def _split_run(K, seed, T, cut):
    """One call of T tokens and two calls of cut + (T - cut) tokens on the
    same inputs (state and cache carried on the device between the two)."""
    inp = inputs.decode_layer(seed, M=2, H=8, T=T)
    tok = inputs.stack_tokens(inp)
    x, w, cache, alpha, beta, S = _device(inp, tok, "f32", "bf16")
    xb, wb, cacheb, alphab, betab, Sb = _device(inp, tok, "f32", "bf16")
    o = K.kda_decode_tokens(x, w, cache, alpha, beta, S)
    oa = K.kda_decode_tokens(xb[:, :cut].contiguous(), wb, cacheb, alphab[:, :cut].contiguous(),
                             betab[:, :cut].contiguous(), Sb)
    ob = K.kda_decode_tokens(xb[:, cut:].contiguous(), wb, cacheb, alphab[:, cut:].contiguous(),
                             betab[:, cut:].contiguous(), Sb)
    torch.cuda.synchronize()
    return o, S, cache, torch.cat([oa, ob], dim=1), Sb, cacheb


def test_tokens_split_equals_whole(K):
    """Two calls of 3 + 5 tokens give the outputs of one call of 8 tokens. The
    chunked kernel groups the tokens of a call into chunks of up to 8, so a
    split that moves a chunk boundary changes the rounding order only: FP32
    agreement to 1e-5, the conv cache bit for bit."""
    o, S, cache, o2, S2, cache2 = _split_run(K, 8200, 8, 3)
    assert rel_err(o2.double().cpu().numpy(), o.double().cpu().numpy()) <= 1e-5
    assert rel_err(to_f64(S2), to_f64(S)) <= 1e-5
    assert torch.equal(cache, cache2)


def test_tokens_split_at_chunk_boundary_is_exact(K):
    """Two calls of 8 + 8 tokens run the same chunks as one call of 16 (the
    FP32 state stored and reloaded in between is exact): bit for bit."""
    o, S, cache, o2, S2, cache2 = _split_run(K, 8210, 16, 8)
    assert torch.equal(o2, o)
    assert torch.equal(S2, S)
    assert torch.equal(cache, cache2)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_tokens_extreme_decay(K, state_dtype):
    """Decays from 1e-30 to exactly 1, mixed per channel and token, over two
    chunks of the chunked kernel (T = 12): its decay ratios are products of
    alphas (never quotients), so nothing overflows; outputs and state match
    the oracle to the usual bar."""
    def extreme(inp, tok):
        rng = np.random.default_rng(9100)
        choices = np.array([1e-30, 1e-3, 0.5, 0.999, 1.0], dtype=np.float32)
        tok["alpha"] = choices[rng.integers(0, len(choices), size=tok["alpha"].shape)]
    o, _, _ = _check(K, 2, 8, 12, state_dtype, seed=90, edit=extreme)
    assert np.all(np.isfinite(o))
