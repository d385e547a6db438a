"""Helpers for the parity tests: move generator inputs onto the device and
run the oracle on the same inputs. Test infrastructure only."""
from __future__ import annotations

import numpy as np

import oracle

#: parity bars (max |gpu - ref| / max |ref|, on o and on S separately)
TOL_F32_STATE = 1e-4
TOL_BF16_STATE = 5e-3


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def bits_to_torch_bf16(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def torch_bf16_to_f64(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32).__lshift__(16) \
        .astype(np.uint32).view(np.float32).astype(np.float64)


def to_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return torch_bf16_to_f64(t)
    return t.detach().cpu().numpy().astype(np.float64)


class DeviceLayer:
    """One KDA layer's inputs resident on the device."""

    def __init__(self, inp: dict, state_dtype: str = "f32", x_dtype: str = "bf16",
                 device="cuda"):
        import torch
        self.inp, self.device = inp, device
        self.x_dtype, self.state_dtype = x_dtype, state_dtype
        self.conv_w = torch.from_numpy(inp["conv_w"]).to(device)
        if x_dtype == "bf16":
            self.cache = bits_to_torch_bf16(inp["cache_bits"], device)
            self.x = [bits_to_torch_bf16(b, device) for b in inp["x_bits"]]
        else:
            self.cache = torch.from_numpy(inp["cache_f32"]).to(device)
            self.x = [torch.from_numpy(v).to(device) for v in inp["x_f32"]]
        S0 = torch.from_numpy(inp["S0"]).to(device)
        # S0 holds BF16-representable values, so this conversion is exact
        self.state = S0.to(torch.bfloat16) if state_dtype == "bf16" else S0
        self.alpha = [torch.from_numpy(a).to(device) for a in inp["alpha"]]
        self.beta = [torch.from_numpy(b).to(device) for b in inp["beta"]]
        M, H, d = inp["M"], inp["H"], inp["d"]
        self.o = torch.empty((M, H, d), dtype=torch.float32, device=device)


def oracle_layer(inp: dict, steps: int | None = None, scale: float = 1.0,
                 heads=None):
    """Run the oracle over the layer's steps; returns (list of o, S, cache).

    heads: optional list of (m, h) pairs; then only those heads' outputs are
    meaningful (the oracle still runs the conv for every channel of the
    streams involved, which is cheap)."""
    T = inp["T"] if steps is None else steps
    S = inp["S0"].astype(np.float64)
    cache = inp["cache_f32"].astype(np.float64)
    outs = []
    for t in range(T):
        o, S, cache = oracle.decode_step(inp["x_f32"][t], inp["conv_w"], cache,
                                         inp["alpha"][t], inp["beta"][t], S, scale=scale)
        outs.append(o)
    return outs, S, cache


def host_workers() -> int:
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def pool_map(fn, tasks):
    """Runs fn over tasks on a thread pool sized to the host's cores. The
    oracle's arithmetic runs in its C library, which ctypes calls without
    the GIL, so the tasks proceed in parallel."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=min(len(tasks), host_workers())) as ex:
        return list(ex.map(fn, tasks))


def oracle_recurrent_all_heads(p: dict, scale: float = 1.0, block: int = 16):
    """The sequential oracle over every (stream, head) of a prefill problem
    (q, k, v, alpha [M, T, H, d], beta [M, T, H], S0 [M, H, d, d]), in tasks
    of `block` heads of one stream. Returns (o [M, T, H, d], S [M, H, d, d])
    in float64."""
    M, T, H, d = p["q"].shape
    block = min(block, H)
    o = np.empty((M, T, H, d), dtype=np.float64)
    S = np.empty((M, H, d, d), dtype=np.float64)

    def task(mh):
        m, h0 = mh
        h1 = min(h0 + block, H)
        sl = (slice(m, m + 1), slice(None), slice(h0, h1))
        oo, SS = oracle.recurrent(p["q"][sl], p["k"][sl], p["v"][sl], p["alpha"][sl],
                                  p["beta"][sl], p["S0"][m:m + 1, h0:h1], scale=scale)
        o[m, :, h0:h1] = oo[0]
        S[m, h0:h1] = SS[0]

    pool_map(task, [(m, h0) for m in range(M) for h0 in range(0, H, block)])
    return o, S


def oracle_prefill_layer_all_heads(p: dict, scale: float = 1.0, norm: bool = True,
                                   block: int = 16):
    """oracle.prefill_layer over every (stream, head) of a layer-prefill
    problem (inputs.prefill_layer_problem), in tasks of `block` heads of one
    stream (each task takes its heads' channels of x, the cache, the conv
    weights and the gate bias). Returns (y [M, T, H, d], S [M, H, d, d],
    cache [M, 3, 3, H*d]) in float64."""
    M, T, three, D = p["x_f32"].shape
    H, d = p["H"], p["d"]
    block = min(block, H)
    y = np.empty((M, T, H, d), dtype=np.float64)
    S = np.empty((M, H, d, d), dtype=np.float64)
    cache = np.empty((M, 3, 3, D), dtype=np.float64)

    def task(mh):
        m, h0 = mh
        h1 = min(h0 + block, H)
        ch = slice(h0 * d, h1 * d)
        hs = slice(h0, h1)
        yy, SS, cc = oracle.prefill_layer(
            p["x_f32"][m:m + 1, :, :, ch], p["conv_w"][:, ch], p["cache_f32"][m:m + 1, :, :, ch],
            p["f"][m:m + 1, :, hs], p["A_log"][hs], p["dt_bias"][ch], p["beta"][m:m + 1, :, hs],
            p["S0"][m:m + 1, hs], scale=scale,
            out_gate=p["out_gate"][m:m + 1, :, hs] if norm else None,
            norm_w=p["norm_w"] if norm else None)
        y[m, :, hs] = yy[0]
        S[m, hs] = SS[0]
        cache[m, :, :, ch] = cc[0]

    pool_map(task, [(m, h0) for m in range(M) for h0 in range(0, H, block)])
    return y, S, cache


def rel_err_per_head(got, ref, head_axes):
    """max |got - ref| / max |ref| taken separately for every index of the
    leading `head_axes` (the remaining axes are one head's tensor). Returns
    an array of errors of shape got.shape[:len(head_axes)] after moving
    head_axes first."""
    got = np.moveaxis(np.asarray(got, dtype=np.float64), head_axes, range(len(head_axes)))
    ref = np.moveaxis(np.asarray(ref, dtype=np.float64), head_axes, range(len(head_axes)))
    k = len(head_axes)
    red = tuple(range(k, got.ndim))
    den = np.max(np.abs(ref), axis=red)
    den = np.where(den > 0, den, 1.0)
    return np.max(np.abs(got - ref), axis=red) / den
