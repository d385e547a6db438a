"""GPU parity of the chunked prefill against the fp64 sequential oracle.

The chunked form must reproduce T sequential steps of the recurrence
("GLM-5.3 deep dive", section 8.2.5): max |gpu - oracle| / max |oracle|
<= 5e-3 on every output and on the final state.
"""
import numpy as np
import pytest

import oracle
from linear_attention_decode_step_gb300 import inputs
from tests.kda_testlib import (bits_to_torch_bf16, oracle_recurrent_all_heads, rel_err,
                               rel_err_per_head)

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


def _device(p, qkv="bf16"):
    dev = "cuda"
    if qkv == "bf16":
        q, k, v = (bits_to_torch_bf16(p[n + "_bits"], dev) for n in ("q", "k", "v"))
    else:
        q, k, v = (torch.from_numpy(p[n]).to(dev) for n in ("q", "k", "v"))
    alpha = torch.from_numpy(p["alpha"]).to(dev)
    beta = torch.from_numpy(p["beta"]).to(dev)
    S = torch.from_numpy(p["S0"]).to(dev).clone()
    return q, k, v, alpha, beta, S


KERNELS = [1, 2]  # KDA_PREFILL_SIMT, KDA_PREFILL_TC


def _run(K, p, qkv="bf16", scale=1.0, kernel=None):
    q, k, v, alpha, beta, S = _device(p, qkv)
    if kernel is None:
        o = K.kda_chunk_prefill(q, k, v, alpha, beta, S, scale=scale)
    else:
        o = K.kda_chunk_prefill_config(q, k, v, alpha, beta, S, scale=scale, kernel=kernel)
    torch.cuda.synchronize()
    assert K.kda_device_error() == K.KDA_OK
    return o.double().cpu().numpy(), S.double().cpu().numpy()


def _oracle(p, scale=1.0, heads=None):
    if heads is None:
        return oracle.recurrent(p["q"], p["k"], p["v"], p["alpha"], p["beta"], p["S0"],
                                scale=scale)
    os_, Ss = [], []
    for (m, h) in heads:
        sl = (slice(m, m + 1), slice(None), slice(h, h + 1))
        o, S = oracle.recurrent(p["q"][sl], p["k"][sl], p["v"][sl], p["alpha"][sl],
                                p["beta"][sl], p["S0"][m:m + 1, h:h + 1], scale=scale)
        os_.append(o[0, :, 0])
        Ss.append(S[0, 0])
    return os_, Ss


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 200])
def test_lengths_and_ragged_chunks(K, T, kernel):
    p = inputs.prefill_problem(4000 + T, M=2, T=T, H=3)
    o, S = _run(K, p, kernel=kernel)
    o_ref, S_ref = _oracle(p)
    assert rel_err(o, o_ref) <= TOL, rel_err(o, o_ref)
    assert rel_err(S, S_ref) <= TOL, rel_err(S, S_ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_fp32_inputs_and_scale(K, kernel):
    p = inputs.prefill_problem(4100, M=1, T=130, H=2)
    scale = 128 ** -0.5
    o, S = _run(K, p, qkv="f32", scale=scale, kernel=kernel)
    o_ref, S_ref = _oracle(p, scale=scale)
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(S, S_ref) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
def test_decay_at_gate_floor(K, kernel):
    """alpha just above e^-5, the floor of the model's gate (section 8.2.3):
    a chunk's summed log-decay reaches about -320, far outside FP32 for a
    single reference point; the 16-token blocks keep every factor finite."""
    p = inputs.prefill_problem(4200, M=1, T=150, H=2)
    rng = np.random.default_rng(4201)
    p["alpha"] = np.exp(-5.0 + 0.05 * rng.random(p["alpha"].shape)).astype(np.float32)
    o, S = _run(K, p, kernel=kernel)
    o_ref, S_ref = _oracle(p)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(S, S_ref) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
def test_slow_decay_long_memory(K, kernel):
    """alpha close to 1 (long memory): the state accumulates over many chunks."""
    p = inputs.prefill_problem(4300, M=1, T=300, H=2, alpha_mean=7.0)
    o, S = _run(K, p, kernel=kernel)
    o_ref, S_ref = _oracle(p)
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(S, S_ref) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
def test_identity_steps_read_state(K, kernel):
    """alpha = 1, beta = 0: the state is unchanged and o_t = S0^T q_t."""
    p = inputs.prefill_problem(4400, M=1, T=70, H=2)
    p["alpha"] = np.ones_like(p["alpha"])
    p["beta"] = np.zeros_like(p["beta"])
    o, S = _run(K, p, kernel=kernel)
    o_ref, S_ref = _oracle(p)
    assert rel_err(S, p["S0"]) <= 1e-6
    assert rel_err(o, o_ref) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
def test_zero_query_and_key_only_decay(K, kernel):
    """q = k = 0 (normalised to 0 through the eps): nothing is written or
    read, so every o_t is exactly 0 and the state is S0 scaled row by row by
    the product of the alphas; across chunk boundaries and a ragged tail."""
    p = inputs.prefill_problem(4800, M=2, T=150, H=3, alpha_mean=4.0)
    for n in ("q", "k"):
        p[n] = np.zeros_like(p[n])
        p[n + "_bits"] = np.zeros_like(p[n + "_bits"])
    o, S = _run(K, p, kernel=kernel)
    assert np.all(o == 0.0)
    o_ref, S_ref = _oracle(p)
    assert rel_err(S, S_ref) <= TOL


@pytest.fixture(scope="module")
def config4():
    """M=4 streams, T=4096 tokens, 64 heads, chunk 64, BF16 q/k/v, FP32 state,
    with the sequential oracle's outputs and final state for every (stream,
    head): 4096 oracle steps per head, run on all host cores."""
    p = inputs.prefill_problem(inputs.layer_seed(inputs.SEED_PREFILL_M4_T4096, 0), M=4, T=4096, H=64)
    o_ref, S_ref = oracle_recurrent_all_heads(p)
    return p, o_ref, S_ref


@pytest.mark.parametrize("kernel", KERNELS)
def test_M4_T4096_every_head(K, config4, kernel):
    """The whole prefill workload on the GPU against 4096 sequential oracle
    steps: every output row and the final state of all 256 (stream, head)
    pairs, each pair to the bar on its own (max error over the pair's o or S
    relative to the pair's largest reference magnitude)."""
    p, o_ref, S_ref = config4
    o, S = _run(K, p, kernel=kernel)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    eo = rel_err_per_head(o, o_ref, (0, 2))      # [M, H] over (T, dv)
    eS = rel_err_per_head(S, S_ref, (0, 1))      # [M, H] over (dk, dv)
    assert eo.shape == (4, 64) and eS.shape == (4, 64)
    assert float(eo.max()) <= TOL, ("o", np.unravel_index(eo.argmax(), eo.shape), float(eo.max()))
    assert float(eS.max()) <= TOL, ("S", np.unravel_index(eS.argmax(), eS.shape), float(eS.max()))
    assert rel_err(o, o_ref) <= TOL and rel_err(S, S_ref) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
def test_mixed_channel_decay_from_the_gate(K, kernel):
    """alpha from the model's forget gate (section 8.2.3): per channel some
    decays sit at the e^-5 floor and others near 1 inside one chunk, so the
    cross-half decay factor of a fast channel underflows while its true
    products with neighbouring tokens do not."""
    p = inputs.prefill_problem(4500, M=1, T=200, H=3)
    gn = inputs.gate_norm_inputs(4501, M=1, H=3, d=128, T=200)
    f = np.stack(gn["f"], axis=1)  # [M, T, H, d]
    p["alpha"] = oracle.forget_gate(f, gn["A_log"], gn["dt_bias"]).astype(np.float32)
    o, S = _run(K, p, kernel=kernel)
    o_ref, S_ref = _oracle(p)
    assert rel_err(o, o_ref) <= TOL, rel_err(o, o_ref)
    assert rel_err(S, S_ref) <= TOL


@pytest.mark.parametrize("M,T,H", [(1, 70, 1), (3, 129, 5)])
def test_odd_shapes(K, M, T, H):
    """One head, and an odd head count with a ragged third chunk: the tensor
    maps of the inputs and the output span every (stream, head) correctly."""
    p = inputs.prefill_problem(4600 + H, M=M, T=T, H=H)
    o, S = _run(K, p, kernel=2)
    o_ref, S_ref = _oracle(p)
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(S, S_ref) <= TOL


def test_output_rows_past_T_untouched(K):
    """O leaves by whole 64-row tensor stores; rows past T must not be
    written (with M > 1 they would be the next stream's). o is handed in as
    the first T rows of a larger buffer filled with a sentinel."""
    p = inputs.prefill_problem(4700, M=1, T=70, H=2)
    q, k, v, alpha, beta, S = _device(p)
    pad = torch.full((1, 128, 2, 128), 12345.0, dtype=torch.float32, device="cuda")
    o = pad[:, :70]
    assert o.is_contiguous()
    K.kda_chunk_prefill_config(q, k, v, alpha, beta, S, o=o, kernel=2)
    torch.cuda.synchronize()
    assert K.kda_device_error() == K.KDA_OK
    assert bool(torch.all(pad[:, 70:] == 12345.0))
    o_ref, _ = _oracle(p)
    assert rel_err(o.double().cpu().numpy(), o_ref) <= TOL


@pytest.mark.parametrize("qkv", ["bf16", "f32"])
def test_pieces_equal_whole_sequences(K, qkv):
    """M = 3 streams x 64 heads (192 sequences, more than the SMs) of 1000
    tokens: the launcher cuts each sequence into pieces of consecutive chunks
    and runs them in rounds, the state passing between pieces in place. Each
    stream's outputs and final state equal, bit for bit, a call of that stream
    alone (64 sequences, fewer than the SMs: one piece each), since a piece
    boundary only stores and reloads the exact FP32 state."""
    p = inputs.prefill_problem(8700, M=3, T=1000, H=64)
    q, k, v, alpha, beta, S = _device(p, qkv)
    o = K.kda_chunk_prefill(q, k, v, alpha, beta, S)
    for m in range(3):
        sl = lambda t: t[m:m + 1].contiguous()
        S1 = sl(torch.from_numpy(p["S0"]).to("cuda"))
        o1 = K.kda_chunk_prefill(sl(q), sl(k), sl(v), sl(alpha), sl(beta), S1)
        torch.cuda.synchronize()
        assert torch.equal(o1[0], o[m]), m
        assert torch.equal(S1[0], S[m]), m
    assert K.kda_device_error() == K.KDA_OK
