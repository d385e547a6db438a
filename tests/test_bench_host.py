"""The measurement arithmetic of bench.py, checked against counts taken from
the tensor layouts (include/kda.h) and from the shapes of the chunked form's
products ("GLM-5.3 deep dive", section 8.2.5), not against the closed forms
bench.py uses. CPU only."""
import numpy as np
import pytest

import bench

H, d = 64, 128
D = H * d


def _nbytes(shape, elem):
    return int(np.prod(shape)) * elem


def test_state_bytes_per_launch():
    for M, dt, s in [(32, "f32", 4), (32, "bf16", 2), (1, "f32", 4)]:
        state = _nbytes((M, H, d, d), s)
        assert bench.state_bytes_per_launch(M, dt) == 2 * state  # read + write


@pytest.mark.parametrize("state_dtype,x_dtype", [("f32", "bf16"), ("bf16", "bf16"), ("f32", "f32")])
def test_decode_algorithmic_bytes_from_layouts(state_dtype, x_dtype):
    M = 32
    s = 4 if state_dtype == "f32" else 2
    x = 4 if x_dtype == "f32" else 2
    total = (2 * _nbytes((M, H, d, d), s)        # state in and out
             + _nbytes((M, 3, D), x)              # pre-conv q, k, v
             + 2 * _nbytes((M, 3, 3, D), x)       # conv cache in and out
             + _nbytes((M, H, d), 4)              # alpha
             + _nbytes((M, H), 4)                 # beta
             + _nbytes((M, H, d), 4)              # o
             + _nbytes((3, D, 4), 4))             # conv weights, shared by the streams
    assert bench.algorithmic_bytes_per_launch(M, state_dtype, x_dtype) == total


def test_headline_roofline_bytes_match_the_profile_figure():
    # the per-launch figure quoted beside the roofline in the decode profile
    assert bench.algorithmic_bytes_per_launch(32, "f32", "bf16") == 281944064


def test_prefill_bytes_from_layouts():
    M, T = 4, 4096
    total = (3 * _nbytes((M, T, H, d), 2)        # q, k, v BF16
             + _nbytes((M, T, H, d), 4)          # alpha
             + _nbytes((M, T, H), 4)             # beta
             + _nbytes((M, T, H, d), 4)          # o
             + 2 * _nbytes((M, H, d, d), 4))     # state in and out
    assert bench.prefill_bytes(M, T, H) == total == 1916796928


@pytest.mark.parametrize("norm", [True, False])
def test_prefill_layer_bytes_from_layouts(norm):
    M, T = 4, 4096
    total = (_nbytes((M, T, 3, D), 2)            # pre-conv x BF16
             + _nbytes((M, T, H, d), 4)          # raw gate input f
             + _nbytes((M, T, H), 4)             # beta
             + (_nbytes((M, T, H, d), 4) if norm else 0)  # output gate
             + _nbytes((M, T, H, d), 4)          # y
             + 2 * _nbytes((M, H, d, d), 4)      # state in and out
             + 2 * _nbytes((M, 3, 3, D), 2))     # conv cache in and out
    assert bench.prefill_layer_bytes(M, T, H, norm=norm) == total


def test_prefill_flops_from_product_shapes():
    """2 m n k per product, over the products of one chunk: A and P scores
    (C x d times d x C), W and U (C x C times C x d), Kd S and Qd S (C x d
    times d x d), the state update (d x C times C x d); ragged last chunks count
    as whole chunks."""
    C = 64
    products = [(C, C, d), (C, C, d), (C, d, C), (C, d, C), (C, d, d), (C, d, d), (d, d, C)]
    per_chunk = sum(2 * m * n * k for m, n, k in products)
    for M, T in [(4, 4096), (2, 1000), (1, 1)]:
        chunks = -(-T // C)
        assert bench.prefill_flops(M, T, H) == per_chunk * M * H * chunks
    assert abs(bench.prefill_flops(4, 4096, H) / 1e9 - 171.8) < 0.05


def test_fp32_peak_from_unit_counts():
    assert abs(bench.fp32_peak_tflops(2070.0) - 152 * 128 * 2 * 2.070e9 / 1e12) < 1e-9
    assert abs(bench.fp32_peak_tflops(None) - bench.fp32_peak_tflops(2070.0)) < 1e-12


def test_tokens_roofline_bound_switches_with_T():
    """A multi-token call moves the state once and does 7 d^2 flops per head
    and token: HBM-bound at small T, ALU-bound once the flops take longer."""
    peak_hbm, mhz = 6778.3, 2070.0
    t_hbm = 2 * 32 * H * d * d * 4 / (peak_hbm * 1e9) * 1e6
    for T in (1, 2, 4, 8, 16, 64):
        t_alu = 7 * d * d * 32 * H * T / (bench.fp32_peak_tflops(mhz) * 1e12) * 1e6
        s = bench.tokens_summary(0.1, 32, T, "f32", peak_hbm, mhz)
        assert s["bound"] == ("hbm" if t_hbm >= t_alu else "alu")
        assert abs(s["roofline_us"] - max(t_hbm, t_alu)) < 1e-9
        assert abs(s["frac_of_roofline"] - max(t_hbm, t_alu) / 100.0) < 1e-12
    assert bench.tokens_summary(0.1, 32, 8, "f32", peak_hbm, mhz)["bound"] == "hbm"
    assert bench.tokens_summary(0.1, 32, 16, "f32", peak_hbm, mhz)["bound"] == "alu"


def test_prefill_summary_fractions():
    s = bench.prefill_summary(1.0, 4, 4096, 6778.3, 1946.6, "k")
    assert abs(s["gb_s"] - 1916796928 / 1e9 / 1e-3) < 1e-6
    assert abs(s["frac_of_measured_hbm"] - s["gb_s"] / 6778.3) < 1e-12
    # the TF32 peak: the measured BF16 peak times the nominal 1.1 / 2.25 PF ratio
    assert abs(s["tf32_peak_tflop_s"] - 1946.6 * 1.1 / 2.25) < 1e-9
    assert s["tf32_peak_kind"] == "measured bf16 x nominal 1.1/2.25"
    assert abs(s["tokens_per_s"] - 4 * 4096 / 1e-3) < 1e-3


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the fp64 oracle on the host cores) prints
    one JSON line with the metric, unit and direction of this library's arm,
    its own e2e object (no host-device bytes) and a cpu_baseline that names
    the oracle and the cores it used. Runs on the CPU in a few seconds."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, check=True, timeout=600, cwd=root)
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["n_gpus"] == 1
    assert line["steps"] == 1 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert cb["sample"]
    assert line["config"]["M"] == 32 and line["config"]["layers"] == 34


def test_traffic_only_for_the_measured_kernel_source(tmp_path, monkeypatch):
    """The roofline's traffic comes from the committed measurement only while
    the decode kernel's source is the one it was taken on, and only for the
    M and state dtype it was taken at."""
    import hashlib
    import json
    src = hashlib.sha256(open(bench.DECODE_SRC, "rb").read()).hexdigest()
    data = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_DATA", str(data))
    assert bench.ncu_traffic_per_launch(32, "f32") is None          # no file
    rows = [{"M": 32, "state_dtype": "f32", "dram_bytes": 2.5e8}]
    data.write_text(json.dumps({"kernel_source_sha256": src, "per_launch": rows}))
    assert bench.ncu_traffic_per_launch(32, "f32") == 2.5e8
    assert bench.ncu_traffic_per_launch(32, "bf16") is None
    assert bench.ncu_traffic_per_launch(8, "f32") is None
    data.write_text(json.dumps({"kernel_source_sha256": "0" * 64, "per_launch": rows}))
    assert bench.ncu_traffic_per_launch(32, "f32") is None          # another source
