"""GPU parity of the decode step with the forget gate fused in front and the
gated RMSNorm fused behind ("GLM-5.3 deep dive" 8.2.3 and 8.2.4 step 7),
against the fp64 oracle: 1e-4 (FP32 state) / 5e-3 (BF16 state) on y and S."""
import numpy as np
import pytest

import oracle
from linear_attention_decode_step_gb300 import inputs
from tests.kda_testlib import (TOL_BF16_STATE, TOL_F32_STATE, DeviceLayer, rel_err, to_f64)

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


def _run(K, M, H, T, state_dtype, x_dtype="bf16", norm=True, seed=0):
    inp = inputs.decode_layer(7000 + seed, M=M, H=H, T=T)
    gn = inputs.gate_norm_inputs(7100 + seed, M=M, H=H, T=T)
    dl = DeviceLayer(inp, state_dtype, x_dtype)
    dev = "cuda"
    A = torch.from_numpy(gn["A_log"]).to(dev)
    b = torch.from_numpy(gn["dt_bias"]).to(dev)
    w = torch.from_numpy(gn["norm_w"]).to(dev)
    S_ref = inp["S0"].astype(np.float64)
    c_ref = inp["cache_f32"].astype(np.float64)
    tol = TOL_BF16_STATE if state_dtype == "bf16" else TOL_F32_STATE
    for t in range(T):
        f = torch.from_numpy(gn["f"][t]).to(dev)
        og = torch.from_numpy(gn["out_gate"][t]).to(dev) if norm else None
        y = K.kda_decode_step_fused(dl.x[t], dl.conv_w, dl.cache, f, A, b, dl.beta[t], dl.state,
                                    out_gate=og, norm_weight=w if norm else None)
        y_ref, S_ref, c_ref = oracle.decode_step_fused(
            inp["x_f32"][t], inp["conv_w"], c_ref, gn["f"][t], gn["A_log"], gn["dt_bias"],
            inp["beta"][t], S_ref, out_gate=gn["out_gate"][t] if norm else None,
            norm_w=gn["norm_w"] if norm else None)
        torch.cuda.synchronize()
        assert rel_err(y.double().cpu().numpy(), y_ref) <= tol, (t, rel_err(y.double().cpu().numpy(), y_ref))
    assert K.kda_device_error() == K.KDA_OK
    assert rel_err(to_f64(dl.state), S_ref) <= tol
    np.testing.assert_array_equal(to_f64(dl.cache), c_ref)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("norm", [True, False])
def test_fused_M32(K, state_dtype, norm):
    _run(K, 32, 64, 2, state_dtype, norm=norm, seed=1)


@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_fused_small_ragged(K, x_dtype):
    _run(K, 3, 5, 3, "f32", x_dtype=x_dtype, seed=2)


def test_fused_rejects_norm_without_weight(K):
    inp = inputs.decode_layer(1, M=1, H=2, T=1)
    dl = DeviceLayer(inp, "f32")
    z = torch.zeros((1, 2, 128), device="cuda")
    with pytest.raises(K.KdaError):
        K.kda_decode_step_fused(dl.x[0], dl.conv_w, dl.cache, z, torch.zeros(2, device="cuda"),
                                torch.zeros(256, device="cuda"), dl.beta[0], dl.state,
                                out_gate=z, norm_weight=None)
