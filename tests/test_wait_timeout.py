"""Failure detection without faulting a GPU.

* Every device-side wait in the library is an mbarrier wait bounded by a
  clock64 budget; on timeout a kernel records an error word (read by
  kda_device_error as KDA_ERR_TIMEOUT) and returns. tests/cuda/wait_probe.cu
  runs the library's own bounded wait on an mbarrier that nothing arrives at,
  with a short budget, and checks that it gives up after about that budget
  and that the context stays usable (a satisfied wait right after succeeds).
* A CUDA error on the host side surfaces as KDA_ERR_CUDA with the cudaError_t
  kept by kda_last_cuda_error: on a machine without a GPU a valid call fails
  at launch (checked on CPU only; with a GPU present the call would launch).
"""
import ctypes
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "cuda", "wait_probe.cu")
CSRC = os.path.join(ROOT, "linear_attention_decode_step_gb300", "csrc")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    so = str(tmp_path_factory.mktemp("wait") / "wait_probe.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I" + CSRC, SRC,
                           "-o", so])
    lib = ctypes.CDLL(so)
    lib.wait_probe_run.argtypes = [ctypes.c_int, ctypes.c_longlong,
                                   ctypes.POINTER(ctypes.c_uint),
                                   ctypes.POINTER(ctypes.c_longlong)]
    lib.wait_probe_run.restype = ctypes.c_int

    def run(mode, budget):
        ok, cycles = ctypes.c_uint(7), ctypes.c_longlong(-1)
        rc = lib.wait_probe_run(mode, budget, ctypes.byref(ok), ctypes.byref(cycles))
        return rc, ok.value, cycles.value
    return run


@pytest.mark.gpu
@pytest.mark.parametrize("budget", [100_000, 2_000_000])
def test_wait_gives_up_after_its_budget(probe, budget):
    rc, ok, cycles = probe(0, budget)
    assert rc == 0
    assert ok == 0
    assert budget <= cycles < budget + 200_000


@pytest.mark.gpu
def test_context_usable_after_a_timeout(probe):
    probe(0, 100_000)
    rc, ok, cycles = probe(1, 100_000)
    assert rc == 0 and ok == 1
    assert cycles < 100_000


def test_cuda_error_surfaces_as_status_without_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("only meaningful (and only safe: the call would launch) without a GPU")
    from linear_attention_decode_step_gb300 import build
    build.build()
    from linear_attention_decode_step_gb300 import kda
    L = kda.lib()
    base, gap = 1 << 40, 1 << 34   # fake, 16-byte aligned, never dereferenced
    st = L.kda_decode_step(base, kda.KDA_BF16, base + gap, base + 2 * gap, kda.KDA_BF16,
                           base + 3 * gap, base + 4 * gap, base + 5 * gap, kda.KDA_F32, 1.0,
                           base + 6 * gap, 2, 4, 128, 128, None)
    assert st == kda.KDA_ERR_CUDA
    assert L.kda_last_cuda_error() != 0
    assert kda.kda_status_string(st) == "KDA_ERR_CUDA"


def test_valid_calls_pass_every_host_check_without_a_gpu():
    """A valid call of every entry point gets past all host-side checks
    (null pointers, sizes, alignment, overlaps) and only then fails, at the
    CUDA runtime, with KDA_ERR_CUDA: the checks reject nothing valid. Fake,
    disjoint, 16-byte aligned addresses are never dereferenced."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("only meaningful (and only safe: the calls would launch) without a GPU")
    from linear_attention_decode_step_gb300 import build
    build.build()
    from linear_attention_decode_step_gb300 import kda
    L = kda.lib()
    A = [(1 << 40) + i * (1 << 34) for i in range(12)]   # disjoint fake buffers
    BF, F = kda.KDA_BF16, kda.KDA_F32
    calls = {
        "kda_conv_step": lambda: L.kda_conv_step(A[0], BF, A[1], A[2], BF, A[3], 2, 512, None),
        "kda_decode_step": lambda: L.kda_decode_step(A[0], BF, A[1], A[2], BF, A[3], A[4], A[5],
                                                     BF, 1.0, A[6], 2, 4, 128, 128, None),
        "kda_decode_step_config": lambda: L.kda_decode_step_config(
            A[0], F, A[1], A[2], F, A[3], A[4], A[5], F, 1.0, A[6], 2, 4, 128, 128,
            kda.KDA_DECODE_CLUSTER, 32, 128, None),
        "kda_decode_step_fused": lambda: L.kda_decode_step_fused(
            A[0], BF, A[1], A[2], BF, A[3], A[4], A[5], -5.0, A[6], A[7], F, 1.0, A[8], A[9],
            1e-5, A[10], 2, 4, 128, 128, None),
        "kda_decode_step_fused (no norm)": lambda: L.kda_decode_step_fused(
            A[0], BF, A[1], A[2], BF, A[3], A[4], A[5], -5.0, A[6], A[7], F, 1.0, None, None,
            1e-5, A[10], 2, 4, 128, 128, None),
        "kda_decode_tokens": lambda: L.kda_decode_tokens(A[0], BF, A[1], A[2], BF, A[3], A[4],
                                                         A[5], F, 1.0, A[6], 2, 5, 4, 128, 128,
                                                         None),
        "kda_chunk_prefill": lambda: L.kda_chunk_prefill(A[0], A[1], A[2], BF, A[3], A[4], A[5],
                                                         A[6], 1.0, 2, 70, 4, 128, 128, 64, None),
        "kda_chunk_prefill_config (SIMT)": lambda: L.kda_chunk_prefill_config(
            A[0], A[1], A[2], F, A[3], A[4], A[5], A[6], 1.0, 2, 70, 4, 128, 128, 64,
            kda.KDA_PREFILL_SIMT, None),
        "kda_prefill_layer": lambda: L.kda_prefill_layer(
            A[0], BF, A[1], A[2], BF, A[3], A[4], A[5], -5.0, A[6], A[7], 1.0, A[8], A[9], 1e-5,
            A[10], 2, 70, 4, 128, 128, 64, None),
        "kda_prefill_layer (no norm)": lambda: L.kda_prefill_layer(
            A[0], F, A[1], A[2], F, A[3], A[4], A[5], -5.0, A[6], A[7], 1.0, None, None, 1e-5,
            A[10], 2, 70, 4, 128, 128, 64, None),
    }
    for name, call in calls.items():
        assert call() == kda.KDA_ERR_CUDA, name
