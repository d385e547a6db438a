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
