"""Python binding of the KDA C ABI (include/kda.h), via ctypes.

Argument marshalling only: every function passes device pointers, sizes and
the current CUDA stream to libkda_gb300.so and raises ``KdaError`` on a
non-OK status. Nothing here computes any part of the method, and there is no
fallback: if the library is missing, loading fails loudly.

Names mirror the C entry points (``kda_conv_step``, ``kda_decode_step``,
``kda_chunk_prefill``...). Tensors are torch CUDA tensors, contiguous, in the
layouts documented in kda.h; PyTorch is used only for device memory and
streams.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

__all__ = [
    "KDA_OK", "KDA_ERR_INVALID_ARG", "KDA_ERR_UNSUPPORTED", "KDA_ERR_ALIGNMENT",
    "KDA_ERR_CUDA", "KDA_ERR_TIMEOUT", "KDA_F32", "KDA_BF16",
    "KDA_DECODE_AUTO", "KDA_DECODE_CLUSTER", "KDA_DECODE_STREAM",
    "KDA_PREFILL_AUTO", "KDA_PREFILL_SIMT", "KDA_PREFILL_TC", "kda_chunk_prefill", "kda_chunk_prefill_config",
    "KdaError", "lib", "load", "library_path", "header_functions",
    "kda_status_string", "kda_last_cuda_error", "kda_version",
    "kda_conv_step", "kda_decode_step", "kda_decode_step_config", "kda_device_error",
    "kda_decode_step_fused", "kda_decode_tokens", "kda_prefill_layer",
]

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED = 0, 1, 2
KDA_ERR_ALIGNMENT, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = 3, 4, 5
KDA_F32, KDA_BF16 = 0, 1
KDA_DECODE_AUTO, KDA_DECODE_CLUSTER, KDA_DECODE_STREAM = 0, 1, 2
KDA_PREFILL_AUTO, KDA_PREFILL_SIMT, KDA_PREFILL_TC = 0, 1, 2

_PKG = os.path.dirname(os.path.abspath(__file__))
_HEADER = os.path.join(os.path.dirname(_PKG), "include", "kda.h")
_lock = threading.Lock()
_lib = None

_V, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

# C signatures (argument types, return type) of every exported entry point
_SIGNATURES = {
    "kda_status_string": ([_I], ctypes.c_char_p),
    "kda_last_cuda_error": ([], _I),
    "kda_version": ([], _I),
    "kda_conv_step": ([_V, _I, _V, _V, _I, _V, _I, _I, _V], _I),
    "kda_decode_step": ([_V, _I, _V, _V, _I, _V, _V, _V, _I, _F, _V,
                         _I, _I, _I, _I, _V], _I),
    "kda_decode_step_config": ([_V, _I, _V, _V, _I, _V, _V, _V, _I, _F, _V,
                                _I, _I, _I, _I, _I, _I, _I, _V], _I),
    "kda_device_error": ([_V], _I),
    "kda_decode_step_fused": ([_V, _I, _V, _V, _I, _V, _V, _V, _F, _V, _V, _I, _F, _V, _V, _F, _V,
                               _I, _I, _I, _I, _V], _I),
    "kda_decode_tokens": ([_V, _I, _V, _V, _I, _V, _V, _V, _I, _F, _V,
                           _I, _I, _I, _I, _I, _V], _I),
    "kda_prefill_layer": ([_V, _I, _V, _V, _I, _V, _V, _V, _F, _V, _V, _F, _V, _V, _F, _V,
                           _I, _I, _I, _I, _I, _I, _V], _I),
    "kda_chunk_prefill": ([_V, _V, _V, _I, _V, _V, _V, _V, _F, _I, _I, _I, _I, _I, _I, _V], _I),
    "kda_chunk_prefill_config": ([_V, _V, _V, _I, _V, _V, _V, _V, _F, _I, _I, _I, _I, _I, _I,
                                  _I, _V], _I),
}


class KdaError(RuntimeError):
    """A KDA entry point returned a non-OK status."""

    def __init__(self, fn: str, status: int):
        self.status = status
        msg = "%s failed: %s" % (fn, _status_name(status))
        if status == KDA_ERR_CUDA:
            msg += " (cudaError %d)" % lib().kda_last_cuda_error()
        super().__init__(msg)


def library_path() -> str:
    return os.path.join(_PKG, "libkda_gb300.so")


def header_functions() -> list[str]:
    """Names of the functions declared in include/kda.h."""
    text = open(_HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def load(path: str) -> ctypes.CDLL:
    """Loads a build of the library from `path` with the C signatures of
    every entry point declared (its own symbols: loaded RTLD_LOCAL)."""
    L = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        f = getattr(L, name)
        f.argtypes, f.restype = args, res
    return L


def lib() -> ctypes.CDLL:
    """The loaded library. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    "libkda_gb300.so is not built (expected at %s); run "
                    "linear_attention_decode_step_gb300.build.build()" % path)
            _lib = load(path)
    return _lib


def _status_name(status: int) -> str:
    return lib().kda_status_string(status).decode()


def kda_status_string(status: int) -> str:
    return _status_name(status)


def kda_last_cuda_error() -> int:
    return lib().kda_last_cuda_error()


def kda_version() -> int:
    return lib().kda_version()


def _check(fn: str, status: int) -> None:
    if status != KDA_OK:
        raise KdaError(fn, status)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KDA_F32
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t.dtype)


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def kda_conv_step(x, conv_w, conv_cache, y=None, stream=None):
    """Short conv + SiLU for one token. x [M,3,D] (bf16|f32), conv_w [3,D,4]
    f32, conv_cache [M,3,3,D] (same dtype as x, updated in place) -> y
    [M,3,D] f32."""
    M, three, D = x.shape
    if y is None:
        y = torch.empty((M, 3, D), dtype=torch.float32, device=x.device)
    st = lib().kda_conv_step(_dev(x, "x"), _dtype_code(x), _dev(conv_w, "conv_w", torch.float32),
                             _dev(conv_cache, "conv_cache"), _dtype_code(conv_cache),
                             _dev(y, "y", torch.float32), M, D, _stream(stream))
    _check("kda_conv_step", st)
    return y


def _decode_args(x, conv_w, conv_cache, alpha, beta, state, o):
    M, H, dk, dv = state.shape
    if o is None:
        o = torch.empty((M, H, dv), dtype=torch.float32, device=state.device)
    args = [_dev(x, "x"), _dtype_code(x), _dev(conv_w, "conv_w", torch.float32),
            _dev(conv_cache, "conv_cache"), _dtype_code(conv_cache),
            _dev(alpha, "alpha", torch.float32), _dev(beta, "beta", torch.float32),
            _dev(state, "state"), _dtype_code(state)]
    return M, H, dk, dv, o, args


def kda_decode_step(x, conv_w, conv_cache, alpha, beta, state, o=None, scale=1.0,
                    stream=None):
    """One fused KDA decode step (see kda.h). state [M,H,128,128] (f32|bf16)
    and conv_cache are updated in place; returns o [M,H,128] f32."""
    M, H, dk, dv, o, args = _decode_args(x, conv_w, conv_cache, alpha, beta, state, o)
    st = lib().kda_decode_step(*args, float(scale), _dev(o, "o", torch.float32),
                               M, H, dk, dv, _stream(stream))
    _check("kda_decode_step", st)
    return o


def kda_decode_step_config(x, conv_w, conv_cache, alpha, beta, state, o=None, scale=1.0,
                           kernel=KDA_DECODE_AUTO, columns=0, threads=0, stream=None):
    """kda_decode_step with an explicit kernel (KDA_DECODE_*) and, for the
    cluster kernel, (columns per CTA, threads per CTA)."""
    M, H, dk, dv, o, args = _decode_args(x, conv_w, conv_cache, alpha, beta, state, o)
    st = lib().kda_decode_step_config(*args, float(scale), _dev(o, "o", torch.float32),
                                      M, H, dk, dv, int(kernel), int(columns), int(threads),
                                      _stream(stream))
    _check("kda_decode_step_config", st)
    return o


def kda_decode_step_fused(x, conv_w, conv_cache, gate_f, A_log, dt_bias, beta, state, y=None,
                          scale=1.0, gate_lower_bound=-5.0, out_gate=None, norm_weight=None,
                          norm_eps=1e-5, stream=None):
    """Decode step with the forget gate fused in front (gate_f replaces alpha)
    and, with out_gate and norm_weight, the gated RMSNorm fused behind.
    Returns y [M,H,128] f32."""
    M, H, dk, dv, y, args = _decode_args(x, conv_w, conv_cache, gate_f, beta, state, y)
    og = _dev(out_gate, "out_gate", torch.float32) if out_gate is not None else None
    nw = _dev(norm_weight, "norm_weight", torch.float32) if norm_weight is not None else None
    st = lib().kda_decode_step_fused(
        args[0], args[1], args[2], args[3], args[4], args[5],
        _dev(A_log, "A_log", torch.float32), _dev(dt_bias, "dt_bias", torch.float32),
        float(gate_lower_bound), args[6], args[7], args[8], float(scale), og, nw, float(norm_eps),
        _dev(y, "y", torch.float32), M, H, dk, dv, _stream(stream))
    _check("kda_decode_step_fused", st)
    return y


def kda_decode_tokens(x, conv_w, conv_cache, alpha, beta, state, o=None, scale=1.0,
                      stream=None):
    """T consecutive decode steps in one call (see kda.h). x [M,T,3,H*128]
    (bf16|f32, pre-conv), alpha [M,T,H,128] f32, beta [M,T,H] f32; state
    [M,H,128,128] (f32|bf16) and conv_cache are updated in place; returns
    o [M,T,H,128] f32."""
    M, H, dk, dv = state.shape
    T = x.shape[1]
    if o is None:
        o = torch.empty((M, T, H, dv), dtype=torch.float32, device=state.device)
    st = lib().kda_decode_tokens(
        _dev(x, "x"), _dtype_code(x), _dev(conv_w, "conv_w", torch.float32),
        _dev(conv_cache, "conv_cache"), _dtype_code(conv_cache),
        _dev(alpha, "alpha", torch.float32), _dev(beta, "beta", torch.float32),
        _dev(state, "state"), _dtype_code(state), float(scale), _dev(o, "o", torch.float32),
        M, T, H, dk, dv, _stream(stream))
    _check("kda_decode_tokens", st)
    return o


def kda_device_error(stream=None) -> int:
    """Waits for the stream and returns (and clears) the device error status:
    KDA_OK or KDA_ERR_TIMEOUT (a bounded device wait gave up)."""
    return lib().kda_device_error(_stream(stream))


def _prefill_args(q, k, v, alpha, beta, state, o):
    M, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.dtype != q.dtype or k.dtype != q.dtype:
        raise ValueError("q, k, v must share shape [M, T, H, 128] and dtype")
    if o is None:
        o = torch.empty((M, T, H, dv), dtype=torch.float32, device=q.device)
    args = [_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dtype_code(q),
            _dev(alpha, "alpha", torch.float32), _dev(beta, "beta", torch.float32),
            _dev(state, "state", torch.float32), _dev(o, "o", torch.float32)]
    return M, T, H, dk, dv, o, args


def kda_chunk_prefill(q, k, v, alpha, beta, state, o=None, scale=1.0, chunk=64, stream=None):
    """Chunked prefill over T tokens (see kda.h). q, k, v [M,T,H,128]
    (bf16|f32, post-conv), alpha [M,T,H,128] f32, beta [M,T,H] f32, state
    [M,H,128,128] f32 updated in place; returns o [M,T,H,128] f32."""
    M, T, H, dk, dv, o, args = _prefill_args(q, k, v, alpha, beta, state, o)
    st = lib().kda_chunk_prefill(*args, float(scale), M, T, H, dk, dv, int(chunk), _stream(stream))
    _check("kda_chunk_prefill", st)
    return o


def kda_chunk_prefill_config(q, k, v, alpha, beta, state, o=None, scale=1.0, chunk=64,
                             kernel=KDA_PREFILL_AUTO, stream=None):
    """kda_chunk_prefill with an explicit kernel (KDA_PREFILL_*)."""
    M, T, H, dk, dv, o, args = _prefill_args(q, k, v, alpha, beta, state, o)
    st = lib().kda_chunk_prefill_config(*args, float(scale), M, T, H, dk, dv, int(chunk),
                                        int(kernel), _stream(stream))
    _check("kda_chunk_prefill_config", st)
    return o


def kda_prefill_layer(x, conv_w, conv_cache, gate_f, A_log, dt_bias, beta, state, y=None,
                      scale=1.0, gate_lower_bound=-5.0, out_gate=None, norm_weight=None,
                      norm_eps=1e-5, chunk=64, stream=None):
    """A KDA layer over a prompt (see kda.h): x [M,T,3,H*128] pre-conv (bf16|f32),
    conv_cache [M,3,3,H*128] (same dtype, updated in place), gate_f [M,T,H,128]
    f32 raw gate input, beta [M,T,H] f32, state [M,H,128,128] f32 updated in
    place; with out_gate and norm_weight the gated RMSNorm is applied.
    Returns y [M,T,H,128] f32."""
    M, T, three, D = x.shape
    H = state.shape[1]
    dk, dv = state.shape[2], state.shape[3]
    if y is None:
        y = torch.empty((M, T, H, dv), dtype=torch.float32, device=x.device)
    og = _dev(out_gate, "out_gate", torch.float32) if out_gate is not None else None
    nw = _dev(norm_weight, "norm_weight", torch.float32) if norm_weight is not None else None
    st = lib().kda_prefill_layer(
        _dev(x, "x"), _dtype_code(x), _dev(conv_w, "conv_w", torch.float32),
        _dev(conv_cache, "conv_cache"), _dtype_code(conv_cache),
        _dev(gate_f, "gate_f", torch.float32), _dev(A_log, "A_log", torch.float32),
        _dev(dt_bias, "dt_bias", torch.float32), float(gate_lower_bound),
        _dev(beta, "beta", torch.float32), _dev(state, "state", torch.float32), float(scale),
        og, nw, float(norm_eps), _dev(y, "y", torch.float32), M, T, H, dk, dv, int(chunk),
        _stream(stream))
    _check("kda_prefill_layer", st)
    return y
