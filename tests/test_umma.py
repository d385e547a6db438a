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


def _with_low_bits(rng, n, low):
    """FP32 values whose 13 bits below the TF32 mantissa are `low`."""
    x = rng.standard_normal(n).astype(np.float32)
    u = (x.view(np.uint32) & np.uint32(0xFFFFE000)) | np.uint32(low)
    return u.view(np.float32)


def _truncated(x):
    return (x.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)


@pytest.mark.parametrize("a_in_tmem", [0, 1])
def test_tf32_operands_are_truncated(probe, a_in_tmem):
    """kind::tf32 reads an FP32 operand by dropping its 13 low mantissa bits
    (no rounding), on both sides and with A from shared or tensor memory.
    The kernels rely on this: adding half a TF32 ulp to an operand before the
    product is then a round to nearest. One-hot rows make D an exact copy of
    the operand as the tensor core sees it."""
    rng = np.random.default_rng(900 + a_in_tmem)
    N, K = 16, 8
    for low in (0x1800, 0x1FFF, 0x0FFF):
        b = _with_low_bits(rng, N, low)
        A = np.zeros((128, K), dtype=np.float32)
        A[:, 0] = 1.0
        B = np.zeros((N, K), dtype=np.float32)
        B[:, 0] = b
        rc, D = probe(A, B, 128, a_in_tmem)
        assert rc == 0
        np.testing.assert_array_equal(D, np.broadcast_to(_truncated(b), (128, N)))
        a = _with_low_bits(rng, 128, low)
        A = np.zeros((128, K), dtype=np.float32)
        A[:, 0] = a
        B = np.zeros((N, K), dtype=np.float32)
        B[:, 0] = 1.0
        rc, D = probe(A, B, 128, a_in_tmem)
        assert rc == 0
        np.testing.assert_array_equal(D, np.broadcast_to(_truncated(a)[:, None], (128, N)))
