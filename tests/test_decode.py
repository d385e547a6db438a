"""GPU parity of the fused decode step against the fp64 oracle.

Every comparison is element by element on the same seeded inputs:
max |gpu - oracle| / max |oracle| <= 1e-4 with FP32 state storage and
<= 5e-3 with BF16 state storage, on o and on S separately; the conv cache is
a pure copy and must match exactly.
"""
import numpy as np
import pytest

import oracle
from linear_attention_decode_step_gb300 import inputs
from tests.kda_testlib import (TOL_BF16_STATE, TOL_F32_STATE, DeviceLayer, pool_map,
                               oracle_layer, rel_err, to_f64)

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


def _tol(state_dtype):
    return TOL_BF16_STATE if state_dtype == "bf16" else TOL_F32_STATE


def _run(K, dl: DeviceLayer, steps, scale=1.0, tile=None, kernel=None, stream_cfg=(0, 0)):
    """tile=(columns, threads) selects the cluster kernel with that split;
    kernel selects a kernel explicitly (stream_cfg = (L2 prefetch, groups)
    for the streaming kernel); neither: the library's choice."""
    outs = []
    for t in range(steps):
        if tile is None and kernel is None:
            K.kda_decode_step(dl.x[t], dl.conv_w, dl.cache, dl.alpha[t], dl.beta[t], dl.state,
                              dl.o, scale=scale)
        else:
            kern = K.KDA_DECODE_CLUSTER if tile is not None else kernel
            cols, thr = tile if tile is not None else stream_cfg
            K.kda_decode_step_config(dl.x[t], dl.conv_w, dl.cache, dl.alpha[t], dl.beta[t],
                                     dl.state, dl.o, scale=scale, kernel=kern, columns=cols,
                                     threads=thr)
        outs.append(dl.o.double().cpu().numpy())
    torch.cuda.synchronize()
    assert K.kda_device_error() == K.KDA_OK
    return outs


def _compare(dl, outs, ref_outs, S_ref, cache_ref, tol):
    for t, (o, r) in enumerate(zip(outs, ref_outs)):
        e = rel_err(o, r)
        assert e <= tol, "o at step %d: rel err %.3e > %.1e" % (t, e, tol)
    e = rel_err(to_f64(dl.state), S_ref)
    assert e <= tol, "S: rel err %.3e > %.1e" % (e, tol)
    np.testing.assert_array_equal(to_f64(dl.cache), cache_ref)


def test_M1_fp32_sixteen_steps(K):
    """M=1, H=64, 128x128, FP32 state, 16 consecutive steps from seed."""
    inp = inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_M1_T16, 0), M=1, T=16)
    dl = DeviceLayer(inp, "f32")
    outs = _run(K, dl, 16)
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, TOL_F32_STATE)


def test_M8_fp32_one_step(K):
    inp = inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_M8, 0), M=8, T=1)
    dl = DeviceLayer(inp, "f32")
    outs = _run(K, dl, 1)
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, TOL_F32_STATE)


def test_M32_bf16_one_step(K):
    """M=32, BF16 state storage, FP32 arithmetic; S0 identical to the FP32 run."""
    inp = inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_M32_BF16, 0), M=32, T=1)
    dl = DeviceLayer(inp, "bf16")
    outs = _run(K, dl, 1)
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, TOL_BF16_STATE)
    # one BF16 rounding of the updated state: within half an ulp of the exact
    # value. BF16 keeps 8 significant bits (7 stored), so half an ulp is at
    # most 2^-8 of the value's magnitude; plus FP32 arithmetic noise.
    got = to_f64(dl.state)
    assert np.all(np.abs(got - S) <= 2.0 ** -8 * np.abs(S) + 1e-6 * np.max(np.abs(S)))


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_M32_one_step(K, state_dtype):
    """The benchmarked workload: M=32, one step, fused conv."""
    inp = inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_STACK, 32), M=32, T=1)
    dl = DeviceLayer(inp, state_dtype)
    outs = _run(K, dl, 1)
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, _tol(state_dtype))


TILES = [(16, 64), (32, 64), (32, 128), (64, 128), (64, 256), (128, 256)]


@pytest.mark.parametrize("kernel", ["cluster", "stream"])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_each_kernel_M32(K, kernel, state_dtype, x_dtype):
    """Both decode kernels at M=32 (2048 heads: many heads per CTA for the
    streaming kernel, so every ring stage is reused), three steps."""
    inp = inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_STACK, 100), M=32, T=3)
    dl = DeviceLayer(inp, state_dtype, x_dtype)
    if kernel == "cluster":
        outs = _run(K, dl, 3, tile=(32, 128))
    else:
        outs = _run(K, dl, 3, kernel=K.KDA_DECODE_STREAM)
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, _tol(state_dtype))


@pytest.mark.parametrize("groups,prefetch", [(1, 0), (2, 0), (2, 3), (1, 2)])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_stream_kernel_ring_configs(K, groups, prefetch, state_dtype):
    """One or two consumer groups on a ring of 3 (FP32) or 5 (BF16) stages,
    with and without L2 prefetch: 2048 heads over the SMs reuse every stage
    many times, so both mbarrier parities and the refill order are exercised."""
    inp = inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_STACK, 200 + groups), M=32, T=2)
    dl = DeviceLayer(inp, state_dtype)
    outs = _run(K, dl, 2, kernel=K.KDA_DECODE_STREAM, stream_cfg=(prefetch, groups))
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, _tol(state_dtype))


@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M,H", [(32, 64), (1, 1), (3, 7), (5, 64), (7, 61)])
def test_packed_bf16_kernel(K, M, H, x_dtype):
    """Four consumer groups of four warps with the BF16 state packed in
    registers (stream kernel, groups = 4): full size, a single head, odd head
    counts and ragged rounds, both input dtypes, two steps."""
    inp = inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_STACK, 400 + M + H), M=M, H=H, T=2)
    dl = DeviceLayer(inp, "bf16", x_dtype)
    outs = _run(K, dl, 2, kernel=K.KDA_DECODE_STREAM, stream_cfg=(0, 4))
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, TOL_BF16_STATE)


def test_packed_kernel_needs_bf16_state(K):
    """groups = 4 exists for BF16 state only: FP32 state is refused."""
    inp = inputs.decode_layer(410, M=2, H=4, T=1)
    dl = DeviceLayer(inp, "f32")
    with pytest.raises(K.KdaError) as err:
        _run(K, dl, 1, kernel=K.KDA_DECODE_STREAM, stream_cfg=(0, 4))
    assert err.value.status == K.KDA_ERR_UNSUPPORTED


@pytest.mark.parametrize("M,H", [(1, 1), (1, 5), (3, 7), (1, 64), (5, 64), (7, 61)])
def test_stream_kernel_small_and_ragged(K, M, H):
    """Streaming kernel with fewer heads than SMs, odd head counts and a
    ragged last round of heads."""
    inp = inputs.decode_layer(300 + M * 100 + H, M=M, H=H, T=2)
    dl = DeviceLayer(inp, "f32")
    outs = _run(K, dl, 2, kernel=K.KDA_DECODE_STREAM)
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, TOL_F32_STATE)


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_every_tile(K, tile, state_dtype, x_dtype):
    inp = inputs.decode_layer(77, M=3, H=5, T=3)
    dl = DeviceLayer(inp, state_dtype, x_dtype)
    outs = _run(K, dl, 3, tile=tile)
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, _tol(state_dtype))


def test_odd_sizes_and_scale(K):
    inp = inputs.decode_layer(5, M=5, H=3, T=4)
    dl = DeviceLayer(inp, "f32")
    scale = 128 ** -0.5
    outs = _run(K, dl, 4, scale=scale)
    ref, S, cache = oracle_layer(inp, scale=scale)
    _compare(dl, outs, ref, S, cache, TOL_F32_STATE)


def test_max_streams_M64(K):
    inp = inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_STACK, 64), M=64, T=1)
    dl = DeviceLayer(inp, "f32")
    outs = _run(K, dl, 1)
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, TOL_F32_STATE)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_identity_step_leaves_state(K, state_dtype):
    """alpha = 1, beta = 0: the state is returned bit for bit and o = S^T q."""
    inp = inputs.decode_layer(6, M=2, H=4, T=1)
    inp["alpha"] = [np.ones_like(inp["alpha"][0])]
    inp["beta"] = [np.zeros_like(inp["beta"][0])]
    dl = DeviceLayer(inp, state_dtype)
    before = dl.state.clone()
    outs = _run(K, dl, 1)
    assert torch.equal(before, dl.state)
    ref, S, cache = oracle_layer(inp)
    assert rel_err(outs[0], ref[0]) <= TOL_F32_STATE


def test_exact_write_beta_one(K):
    """beta = 1: after the step, reading with the normalised key returns v
    (section 8.2.3), checked against the oracle's state."""
    inp = inputs.decode_layer(8, M=2, H=4, T=1)
    inp["beta"] = [np.ones_like(inp["beta"][0])]
    dl = DeviceLayer(inp, "f32")
    outs = _run(K, dl, 1)
    ref, S, cache = oracle_layer(inp)
    _compare(dl, outs, ref, S, cache, TOL_F32_STATE)


def test_zero_input_degenerate(K):
    """All-zero pre-conv input and cache: q = k = 0 after the conv, so the
    update only fades the state and o = 0."""
    inp = inputs.decode_layer(9, M=2, H=4, T=1)
    inp["x_bits"] = [np.zeros_like(inp["x_bits"][0])]
    inp["x_f32"] = [np.zeros_like(inp["x_f32"][0])]
    inp["cache_bits"] = np.zeros_like(inp["cache_bits"])
    inp["cache_f32"] = np.zeros_like(inp["cache_f32"])
    dl = DeviceLayer(inp, "f32")
    outs = _run(K, dl, 1)
    ref, S, cache = oracle_layer(inp)
    assert np.all(outs[0] == 0.0)
    _compare(dl, outs, ref, S, cache, TOL_F32_STATE)


@pytest.mark.parametrize("M", [8, 32])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_34_layer_stack_under_cuda_graph(K, state_dtype, M):
    """34 independent layers launched as one captured CUDA graph per token,
    exactly as the bench launches them (programmatic dependent launch between
    layers, each layer's state prefetched into L2 before it waits for the
    previous one), at M=8 and at the benchmarked M=32, for two tokens (two
    replays, the state carried). Each token of every layer is checked against
    one oracle step taken from the state the GPU had stored before it (with
    BF16 storage that state is rounded, and the bar holds per step; two steps
    against an unrounded reference would compound two roundings)."""
    L, T = 34, 2
    layers = [DeviceLayer(inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_STACK, l), M=M, T=T),
                          state_dtype) for l in range(L)]
    outs = [[torch.empty_like(dl.o) for _ in range(T)] for dl in layers]
    s = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(s):
        for t in range(T):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for dl, ol in zip(layers, outs):
                    K.kda_decode_step(dl.x[t], dl.conv_w, dl.cache, dl.alpha[t], dl.beta[t],
                                      dl.state, ol[t])
            graphs.append(g)
    states = []  # the state each layer held before token t, as stored (host copies)
    for t, g in enumerate(graphs):
        torch.cuda.synchronize()
        states.append([dl.state.cpu() for dl in layers])
        g.replay()
    torch.cuda.synchronize()
    assert K.kda_device_error() == K.KDA_OK
    tol = _tol(state_dtype)

    def check(l):
        dl, inp = layers[l], layers[l].inp
        cache = inp["cache_f32"].astype(np.float64)
        for t in range(T):
            o_ref, S_ref, cache = oracle.decode_step(inp["x_f32"][t], inp["conv_w"], cache,
                                                     inp["alpha"][t], inp["beta"][t],
                                                     to_f64(states[t][l]))
            e = rel_err(outs[l][t].double().cpu().numpy(), o_ref)
            assert e <= tol, "layer %d token %d: o rel err %.3e" % (l, t, e)
            got = to_f64(states[t + 1][l] if t + 1 < T else dl.state)
            e = rel_err(got, S_ref)
            assert e <= tol, "layer %d token %d: S rel err %.3e" % (l, t, e)
        np.testing.assert_array_equal(to_f64(dl.cache), cache)
    pool_map(check, list(range(L)))


@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_conv_step(K, x_dtype):
    inp = inputs.decode_layer(10, M=3, H=64, T=2)
    dl = DeviceLayer(inp, "f32", x_dtype)
    cache = inp["cache_f32"].astype(np.float64)
    for t in range(2):
        y = K.kda_conv_step(dl.x[t], dl.conv_w, dl.cache)
        y_ref, cache = oracle.conv_step(inp["x_f32"][t], inp["conv_w"], cache)
        torch.cuda.synchronize()
        assert rel_err(y.double().cpu().numpy(), y_ref) <= 1e-6
        np.testing.assert_array_equal(to_f64(dl.cache), cache)
