"""The library's tcgen05 wrappers (descriptors, MMA issue, TMEM loads and
stores) against numpy: D = A B^T on the tensor cores, kind::tf32.

Builds tests/cuda/umma_probe.cu (which includes the library's own
kda_umma.cuh / kda_ptx.cuh) into a temporary library with nvcc.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "cuda", "umma_probe.cu")
CSRC = os.path.join(ROOT, "linear_attention_decode_step_gb300", "csrc")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    so = str(tmp_path_factory.mktemp("umma") / "umma_probe.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I" + CSRC, SRC,
                           "-o", so])
    lib = ctypes.CDLL(so)
    P = ctypes.POINTER(ctypes.c_float)
    lib.umma_probe_run.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int]
    lib.umma_probe_run.restype = ctypes.c_int

    def run(A, B, M, mode):
        N, K = B.shape
        A = np.ascontiguousarray(A, dtype=np.float32)
        B = np.ascontiguousarray(B, dtype=np.float32)
        D = np.zeros((128, N), dtype=np.float32)
        p = lambda a: a.ctypes.data_as(P)
        rc = lib.umma_probe_run(p(A), p(B), p(D), M, N, K, mode)
        return rc, D
    return run


def _tf32_err(D, ref):
    return np.max(np.abs(D - ref)) / np.max(np.abs(ref))


@pytest.mark.parametrize("N,K", [(64, 32), (128, 64), (16, 8)])
@pytest.mark.parametrize("a_in_tmem", [0, 1])
def test_m128_product(probe, N, K, a_in_tmem):
    rng = np.random.default_rng(N * 100 + K + a_in_tmem)
    A = rng.standard_normal((128, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    rc, D = probe(A, B, 128, a_in_tmem)
    assert rc == 0
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    assert _tf32_err(D, ref) < 4e-3   # TF32 operands: 10-bit mantissa
