"""The C-ABI library builds, loads, exports every symbol include/kda.h
declares, and rejects bad arguments on the host before touching the device.

These run without a GPU: every call below returns from the host-side checks
(fake but aligned, non-overlapping addresses are never dereferenced).
"""
import ctypes
import subprocess

import pytest

from linear_attention_decode_step_gb300 import build as kbuild


@pytest.fixture(scope="module")
def K():
    kbuild.build()
    from linear_attention_decode_step_gb300 import kda
    return kda


def test_header_symbols_exported(K):
    names = K.header_functions()
    assert {"kda_conv_step", "kda_decode_step", "kda_status_string"} <= set(names)
    L = K.lib()
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", K.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert set(names) <= exported
    # every declared function has a binding signature and a public wrapper
    assert set(names) <= set(K._SIGNATURES)
    assert set(names) <= set(K.__all__)
    for n in names:
        assert callable(getattr(K, n)), n


def test_status_strings(K):
    assert K.kda_status_string(0) == "KDA_OK"
    assert K.kda_status_string(4) == "KDA_ERR_CUDA"
    assert K.kda_status_string(99) == "KDA_ERR_UNKNOWN"
    assert K.kda_version() >= 100
    assert K.kda_last_cuda_error() == 0


# fake device addresses: 16-byte aligned, far apart (never dereferenced)
BASE = 1 << 40
GAP = 1 << 34


def _decode_call(K, **over):
    a = dict(x=BASE, xd=K.KDA_BF16, w=BASE + GAP, cache=BASE + 2 * GAP, cd=K.KDA_BF16,
             alpha=BASE + 3 * GAP, beta=BASE + 4 * GAP, state=BASE + 5 * GAP,
             sd=K.KDA_F32, scale=1.0, o=BASE + 6 * GAP, M=4, H=64, dk=128, dv=128)
    a.update(over)
    return K.lib().kda_decode_step(a["x"], a["xd"], a["w"], a["cache"], a["cd"], a["alpha"],
                                   a["beta"], a["state"], a["sd"], a["scale"], a["o"],
                                   a["M"], a["H"], a["dk"], a["dv"], None)


@pytest.mark.parametrize("field", ["x", "w", "cache", "alpha", "beta", "state", "o"])
def test_decode_null_pointer(K, field):
    assert _decode_call(K, **{field: None}) == K.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("field", ["x", "w", "cache", "alpha", "beta", "state", "o"])
def test_decode_misaligned(K, field):
    base = {"x": BASE, "w": BASE + GAP, "cache": BASE + 2 * GAP, "alpha": BASE + 3 * GAP,
            "beta": BASE + 4 * GAP, "state": BASE + 5 * GAP, "o": BASE + 6 * GAP}[field]
    assert _decode_call(K, **{field: base + 4}) == K.KDA_ERR_ALIGNMENT


@pytest.mark.parametrize("over,status", [
    (dict(M=0), 1), (dict(H=0), 1), (dict(M=-3), 1), (dict(dk=0), 1),
    (dict(dk=64), 2), (dict(dv=64), 2), (dict(dk=256, dv=256), 2),
    (dict(M=70000), 2), (dict(M=65535, H=65535), 2),  # M * H beyond 2^30
    (dict(xd=7), 1), (dict(sd=-1), 1), (dict(cd=5), 1),
    (dict(cd=0), 2),                       # cache dtype must equal x dtype
    (dict(o=BASE + 5 * GAP + 1024), 1),    # o inside the state buffer
    (dict(cache=BASE + 5 * GAP), 1),       # cache aliases the state
    (dict(o=BASE + 3 * GAP + 64), 1),      # o inside alpha
    (dict(o=BASE + 4 * GAP + 16), 1),      # o inside beta
    (dict(state=BASE + 16), 1),            # state overlaps x
    (dict(cache=BASE + GAP + 32), 1),      # cache inside the conv weights
])
def test_decode_rejects(K, over, status):
    assert _decode_call(K, **over) == status


def test_decode_unsupported_config(K):
    L = K.lib()
    args = (BASE, 1, BASE + GAP, BASE + 2 * GAP, 1, BASE + 3 * GAP, BASE + 4 * GAP,
            BASE + 5 * GAP, 0, 1.0, BASE + 6 * GAP, 4, 64, 128, 128)
    assert L.kda_decode_step_config(*args, K.KDA_DECODE_CLUSTER, 48, 96, None) \
        == K.KDA_ERR_UNSUPPORTED
    assert L.kda_decode_step_config(*args, 7, 0, 0, None) == K.KDA_ERR_INVALID_ARG
    # streaming kernel: L2 prefetch distance beyond 16, or 3 consumer groups
    assert L.kda_decode_step_config(*args, K.KDA_DECODE_STREAM, 17, 0, None) \
        == K.KDA_ERR_UNSUPPORTED
    assert L.kda_decode_step_config(*args, K.KDA_DECODE_STREAM, 0, 3, None) \
        == K.KDA_ERR_UNSUPPORTED


def test_conv_rejects(K):
    L = K.lib()
    ok = dict(x=BASE, xd=1, w=BASE + GAP, c=BASE + 2 * GAP, cd=1, y=BASE + 3 * GAP, M=2, D=8192)

    def call(**o):
        a = dict(ok)
        a.update(o)
        return L.kda_conv_step(a["x"], a["xd"], a["w"], a["c"], a["cd"], a["y"],
                               a["M"], a["D"], None)
    assert call(x=None) == K.KDA_ERR_INVALID_ARG
    assert call(y=BASE + 3 * GAP + 2) == K.KDA_ERR_ALIGNMENT
    assert call(M=0) == K.KDA_ERR_INVALID_ARG
    assert call(cd=0) == K.KDA_ERR_UNSUPPORTED
    assert call(c=BASE + 16) == K.KDA_ERR_INVALID_ARG          # cache overlaps x
    assert call(c=BASE + GAP + 16) == K.KDA_ERR_INVALID_ARG    # cache inside the weights
    assert call(y=BASE + 16) == K.KDA_ERR_INVALID_ARG   # y overlaps x


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from linear_attention_decode_step_gb300 import kda
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(kda, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        kda.lib()


def _prefill_call(K, **over):
    a = dict(q=BASE, k=BASE + GAP, v=BASE + 2 * GAP, qd=K.KDA_BF16, alpha=BASE + 3 * GAP,
             beta=BASE + 4 * GAP, state=BASE + 5 * GAP, o=BASE + 6 * GAP, scale=1.0,
             M=4, T=4096, H=64, dk=128, dv=128, chunk=64)
    a.update(over)
    return K.lib().kda_chunk_prefill(a["q"], a["k"], a["v"], a["qd"], a["alpha"], a["beta"],
                                     a["state"], a["o"], a["scale"], a["M"], a["T"], a["H"],
                                     a["dk"], a["dv"], a["chunk"], None)


@pytest.mark.parametrize("over,status", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(state=None), 1), (dict(T=0), 1),
    (dict(M=0), 1), (dict(chunk=0), 1), (dict(qd=3), 1),
    (dict(chunk=32), 2), (dict(dk=64), 2), (dict(dv=256), 2), (dict(H=70000), 2),
    (dict(M=40000, H=40000), 2),           # M * H beyond 2^30
    (dict(alpha=BASE + 3 * GAP + 8), 3), (dict(o=BASE + 6 * GAP + 4), 3),
    (dict(o=BASE + 16), 1),                 # o overlaps q
    (dict(state=BASE + 3 * GAP + 64), 1),   # state inside alpha
])
def test_prefill_rejects(K, over, status):
    assert _prefill_call(K, **over) == status


def _tokens_call(K, **over):
    a = dict(x=BASE, xd=K.KDA_BF16, w=BASE + GAP, cache=BASE + 2 * GAP, cd=K.KDA_BF16,
             alpha=BASE + 3 * GAP, beta=BASE + 4 * GAP, state=BASE + 5 * GAP,
             sd=K.KDA_F32, scale=1.0, o=BASE + 6 * GAP, M=4, T=8, H=64, dk=128, dv=128)
    a.update(over)
    return K.lib().kda_decode_tokens(a["x"], a["xd"], a["w"], a["cache"], a["cd"], a["alpha"],
                                     a["beta"], a["state"], a["sd"], a["scale"], a["o"],
                                     a["M"], a["T"], a["H"], a["dk"], a["dv"], None)


@pytest.mark.parametrize("over,status", [
    (dict(T=0), 1), (dict(T=-1), 1), (dict(x=None), 1), (dict(o=None), 1),
    (dict(M=0), 1), (dict(dk=64), 2), (dict(cd=0), 2), (dict(alpha=BASE + 3 * GAP + 8), 3),
    # o spans M*T*H*128 floats: its end (4*8*64*128*4 bytes = 1 MiB) reaches the state
    (dict(o=BASE + 5 * GAP - (1 << 20) + 16), 1),
])
def test_tokens_rejects(K, over, status):
    assert _tokens_call(K, **over) == status


def _layer_call(K, **over):
    a = dict(x=BASE, xd=K.KDA_BF16, w=BASE + GAP, cache=BASE + 2 * GAP, cd=K.KDA_BF16,
             f=BASE + 3 * GAP, A=BASE + 4 * GAP, bias=BASE + 5 * GAP, lb=-5.0,
             beta=BASE + 6 * GAP, state=BASE + 7 * GAP, scale=1.0, og=None, nw=None,
             neps=1e-5, y=BASE + 8 * GAP, M=4, T=4096, H=64, dk=128, dv=128, chunk=64)
    a.update(over)
    return K.lib().kda_prefill_layer(a["x"], a["xd"], a["w"], a["cache"], a["cd"], a["f"], a["A"],
                                     a["bias"], a["lb"], a["beta"], a["state"], a["scale"],
                                     a["og"], a["nw"], a["neps"], a["y"], a["M"], a["T"], a["H"],
                                     a["dk"], a["dv"], a["chunk"], None)


@pytest.mark.parametrize("over,status", [
    (dict(x=None), 1), (dict(f=None), 1), (dict(A=None), 1), (dict(T=0), 1), (dict(chunk=32), 2),
    (dict(dk=64), 2), (dict(cd=0), 2), (dict(og=BASE + 9 * GAP), 1),  # out_gate without weight
    (dict(f=BASE + 3 * GAP + 4), 3), (dict(state=BASE + 2 * GAP), 1),  # state aliases the cache
    (dict(y=BASE + GAP + 16), 1),          # y inside the conv weights
    (dict(cache=BASE + 4 * GAP), 1),       # cache aliases A_log
    (dict(state=BASE + 5 * GAP + 16), 1),  # state overlaps dt_bias
])
def test_layer_rejects(K, over, status):
    assert _layer_call(K, **over) == status


def _fused_call(K, **over):
    a = dict(x=BASE, xd=K.KDA_BF16, w=BASE + GAP, cache=BASE + 2 * GAP, cd=K.KDA_BF16,
             f=BASE + 3 * GAP, A=BASE + 4 * GAP, bias=BASE + 5 * GAP, lb=-5.0,
             beta=BASE + 6 * GAP, state=BASE + 7 * GAP, sd=K.KDA_F32, scale=1.0,
             og=BASE + 8 * GAP, nw=BASE + 9 * GAP, neps=1e-5, y=BASE + 10 * GAP,
             M=4, H=64, dk=128, dv=128)
    a.update(over)
    return K.lib().kda_decode_step_fused(a["x"], a["xd"], a["w"], a["cache"], a["cd"], a["f"],
                                         a["A"], a["bias"], a["lb"], a["beta"], a["state"],
                                         a["sd"], a["scale"], a["og"], a["nw"], a["neps"],
                                         a["y"], a["M"], a["H"], a["dk"], a["dv"], None)


@pytest.mark.parametrize("over,status", [
    (dict(A=None), 1), (dict(bias=None), 1), (dict(nw=None), 1),  # out_gate without weight
    (dict(og=BASE + 8 * GAP + 4), 3), (dict(dk=64), 2),
    (dict(y=BASE + 4 * GAP), 1),           # y aliases A_log
    (dict(cache=BASE + 5 * GAP + 16), 1),  # cache overlaps dt_bias
    (dict(state=BASE + 9 * GAP), 1),       # state aliases the norm weight
    (dict(y=BASE + 8 * GAP + 16), 1),      # y overlaps the output gate
    (dict(y=BASE + 3 * GAP + 16), 1),      # y overlaps the gate input
])
def test_fused_rejects(K, over, status):
    assert _fused_call(K, **over) == status


def test_plain_c_caller(K, tmp_path):
    """The header compiles as strict C99 (gcc -pedantic -Werror, no C++ or
    CUDA headers) and a C program linked with the library gets the documented
    statuses from the host-side checks (tests/c/abi_caller.c)."""
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(K.library_path())
    exe = tmp_path / "abi_caller"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(root, "include"),
                    os.path.join(root, "tests", "c", "abi_caller.c"),
                    "-L", libdir, "-lkda_gb300", "-Wl,-rpath," + libdir, "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "abi_caller: ok"
