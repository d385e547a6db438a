#!/usr/bin/env python3
"""KDA decode benchmark on GB300: state GB/s and ms/layer at M=32, FP32 state.

One step is one token through a 34-layer KDA decode stack (GLM-5.3-Flash has
34 KDA layers): 34 launches of the fused decode kernel (conv + SiLU, L2 norm,
Eq. 1 update, readout), each on its own layer's state and conv cache, with
M = 32 streams x 64 heads x 128 x 128 FP32 state (134 MB per layer; 4.6 GB
touched per step, so every layer's state comes from HBM, not L2).

Printed (rank 0, one JSON line): value = state GB/s (2 * state bytes per
layer per step / time), ms_per_step, ms_per_layer, the roofline of the
decode kernel against the measured HBM peak, an end-to-end number through the
public API with per-step host<->device copies, the SM clocks seen during the
timed region, and the fp64 CPU oracle timed on a bounded sample.

  python bench.py [--gpus N --steps K --warmup W]        this library
  python bench.py --impl reference [...]                  the CPU oracle
Multi-GPU (torchrun, one rank per GPU): independent replicas, weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_decode_step_gb300 import replicas  # noqa: E402

METRIC = "KDA decode state GB/s & ms/layer at M=32 FP32 (fraction of GB300 HBM peak)"
UNIT = "GB/s"
H, DH = 64, 128
LAYERS = 34
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "linear_attention_decode_step_gb300", "csrc")
# the kernel kda_decode_step runs for this workload (M*H >= 512 heads) and its source
DECODE_KERNEL = "kda_decode_stream_kernel"
DECODE_SRC = os.path.join(CSRC, "kda_decode_stream.cu")
# measured DRAM traffic per launch of the decode kernel (ncu, several consecutive
# launches of a small stack), keyed by the SHA-256 of the kernel's source
TRAFFIC_DATA = os.path.join(ROOT, "profiles", "kda_decode_traffic.json")


# --------------------------------------------------------------------------- sizes
def dtype_size(name: str) -> int:
    return 2 if name == "bf16" else 4


def state_bytes_per_launch(M: int, state_dtype: str) -> int:
    """State read + write of one layer: 2 * M * H * dk * dv * sizeof(state)."""
    return 2 * M * H * DH * DH * dtype_size(state_dtype)


def algorithmic_bytes_per_launch(M: int, state_dtype: str, x_dtype: str) -> int:
    """Every byte one launch must move at least once.

    Per (stream, head): state read + write 2*dk*dv*s, pre-conv q/k/v 3*d*x,
    conv cache read + write 2*9*d*x, alpha 4*d, beta 4, o 4*d. Per launch:
    conv weights 3*H*d*4*4 (shared by all streams).
    """
    s, x = dtype_size(state_dtype), dtype_size(x_dtype)
    per_unit = 2 * DH * DH * s + 3 * DH * x + 18 * DH * x + 4 * DH + 4 + 4 * DH
    return M * H * per_unit + 3 * H * DH * 16


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic_per_launch(M: int, state_dtype: str):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch of the decode
    kernel at this M and state dtype, from the committed measurement, if it
    was taken on the current kernel source (else None)."""
    try:
        with open(TRAFFIC_DATA) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    src = hashlib.sha256(open(DECODE_SRC, "rb").read()).hexdigest()
    if data.get("kernel_source_sha256") != src:
        return None
    for row in data.get("per_launch", []):
        if row.get("M") == M and row.get("state_dtype") == state_dtype:
            return float(row["dram_bytes"])
    return None


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id, self.proc, self.path = gpu_id, None, None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["--id=" + self.gpu_id]
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        for line in open(self.path):
            f = [t.strip() for t in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(torch, dev) -> str | None:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# --------------------------------------------------------------------------- workload
class DecodeStack:
    """L independent KDA layers resident on one GPU, with pinned host
    mirrors of the per-step inputs and outputs for the end-to-end leg."""

    def __init__(self, torch, kda, inputs, M, L, state_dtype, x_dtype, device, seed_space=None,
                 kernel=0, columns=0, threads=0, replicate=False, rank=0):
        """replicate=True draws one layer's inputs and copies them into every
        layer's buffers (used by the sweep, where only timing matters)."""
        self.torch, self.kda, self.M, self.L = torch, kda, M, L
        self.state_dtype, self.x_dtype = state_dtype, x_dtype
        if seed_space is None:
            seed_space = inputs.SEED_DECODE_STACK
        D = H * DH
        xt = torch.bfloat16 if x_dtype == "bf16" else torch.float32
        st = torch.bfloat16 if state_dtype == "bf16" else torch.float32
        # per-step inputs of all layers in one buffer each (one copy per step);
        # two sets, so the end-to-end leg can copy step k+1 in while step k runs
        self.xs = [torch.empty((L, M, 3, D), dtype=xt, device=device) for _ in range(2)]
        self.alphas = [torch.empty((L, M, H, DH), dtype=torch.float32, device=device)
                       for _ in range(2)]
        self.betas = [torch.empty((L, M, H), dtype=torch.float32, device=device) for _ in range(2)]
        self.os = [torch.empty((L, M, H, DH), dtype=torch.float32, device=device) for _ in range(2)]
        self.x, self.alpha, self.beta, self.o = self.xs[0], self.alphas[0], self.betas[0], self.os[0]
        self.conv_w, self.cache, self.state = [], [], []
        self.host0 = None
        for l in range(L):
            if l == 0 or not replicate:
                inp = inputs.decode_layer(replicas.rank_layer_seed(seed_space, l, rank), M=M, T=1)
            if l == 0:
                self.host0 = inp
            if x_dtype == "bf16":
                self.x[l].copy_(torch.from_numpy(inp["x_bits"][0].view(np.int16)).view(torch.bfloat16))
                cache = torch.from_numpy(inp["cache_bits"].view(np.int16)).to(device).view(torch.bfloat16)
            else:
                self.x[l].copy_(torch.from_numpy(inp["x_f32"][0]))
                cache = torch.from_numpy(inp["cache_f32"]).to(device)
            self.alpha[l].copy_(torch.from_numpy(inp["alpha"][0]))
            self.beta[l].copy_(torch.from_numpy(inp["beta"][0]))
            self.conv_w.append(torch.from_numpy(inp["conv_w"]).to(device))
            self.cache.append(cache)
            self.state.append(torch.from_numpy(inp["S0"]).to(device).to(st))
        self.xs[1].copy_(self.x)
        self.alphas[1].copy_(self.alpha)
        self.betas[1].copy_(self.beta)
        self.x_h = self.x.cpu().pin_memory()
        self.alpha_h = self.alpha.cpu().pin_memory()
        self.beta_h = self.beta.cpu().pin_memory()
        self.o_h = [torch.empty(self.o.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
        self.stream = torch.cuda.Stream(device=device)
        self.lib = kda.lib()
        sp = self.stream.cuda_stream
        xd = kda.KDA_BF16 if x_dtype == "bf16" else kda.KDA_F32
        sd = kda.KDA_BF16 if state_dtype == "bf16" else kda.KDA_F32
        # marshalled C-ABI arguments of each layer's decode call, per buffer set
        self.kernel = (kernel, columns, threads)
        self.fn = self.lib.kda_decode_step if kernel == 0 else self.lib.kda_decode_step_config
        tail = (sp,) if kernel == 0 else (kernel, columns, threads, sp)
        self.calls = [[(self.xs[b][l].data_ptr(), xd, self.conv_w[l].data_ptr(),
                        self.cache[l].data_ptr(), xd, self.alphas[b][l].data_ptr(),
                        self.betas[b][l].data_ptr(), self.state[l].data_ptr(), sd, 1.0,
                        self.os[b][l].data_ptr(), M, H, DH, DH) + tail for l in range(L)]
                      for b in range(2)]

    def launch(self, l: int, b: int = 0):
        st = self.fn(*self.calls[b][l])
        if st != 0:
            raise self.kda.KdaError("kda_decode_step", st)

    def step(self, b: int = 0):
        for l in range(self.L):
            self.launch(l, b)

    def copy_in(self, b: int = 0):
        self.xs[b].copy_(self.x_h, non_blocking=True)
        self.alphas[b].copy_(self.alpha_h, non_blocking=True)
        self.betas[b].copy_(self.beta_h, non_blocking=True)

    def copy_out(self, b: int = 0):
        self.o_h[b].copy_(self.os[b], non_blocking=True)

    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.x_h, self.alpha_h, self.beta_h))

    def d2h_bytes(self) -> int:
        return self.o_h[0].numel() * self.o_h[0].element_size()


def time_device(stack: DecodeStack, K: int, W: int, barrier):
    """K steps with inputs resident. One step (L launches of the decode
    kernel through the C ABI) is captured once as a CUDA graph and replayed;
    an event pair brackets every replay. Returns (total ms, per-step ms)."""
    torch = stack.torch
    with torch.cuda.stream(stack.stream):
        stack.step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stack.stream):
            stack.step()
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
        barrier()
        torch.cuda.synchronize()
        ev[0].record(stack.stream)
        for k in range(K):
            g.replay()
            ev[k + 1].record(stack.stream)
        torch.cuda.synchronize()
        barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev[:-1], ev[1:])]
    return ev[0].elapsed_time(ev[-1]), step_ms


def time_fused(stack: DecodeStack, inputs, K: int, W: int):
    """The same stack through kda_decode_step_fused: forget gate fused in
    front (raw gate input f per layer instead of alpha) and gated RMSNorm
    fused behind (output gate per layer). Graph of L launches, K replays."""
    torch = stack.torch
    L, M = stack.L, stack.M
    dev = stack.x.device
    gn = inputs.gate_norm_inputs(9, M=M, H=H, T=1)
    A = torch.from_numpy(gn["A_log"]).to(dev)
    b = torch.from_numpy(gn["dt_bias"]).to(dev)
    w = torch.from_numpy(gn["norm_w"]).to(dev)
    f = torch.from_numpy(gn["f"][0]).to(dev).unsqueeze(0).repeat(L, 1, 1, 1).contiguous()
    og = torch.from_numpy(gn["out_gate"][0]).to(dev).unsqueeze(0).repeat(L, 1, 1, 1).contiguous()
    xd = stack.calls[0][0][1]
    sd = stack.calls[0][0][8]
    sp = stack.stream.cuda_stream
    fn = stack.lib.kda_decode_step_fused
    calls = [(stack.x[l].data_ptr(), xd, stack.conv_w[l].data_ptr(), stack.cache[l].data_ptr(), xd,
              f[l].data_ptr(), A.data_ptr(), b.data_ptr(), -5.0, stack.beta[l].data_ptr(),
              stack.state[l].data_ptr(), sd, 1.0, og[l].data_ptr(), w.data_ptr(), 1e-5,
              stack.o[l].data_ptr(), M, H, DH, DH, sp) for l in range(L)]

    def step():
        for c in calls:
            st = fn(*c)
            if st != 0:
                raise stack.kda.KdaError("kda_decode_step_fused", st)
    with torch.cuda.stream(stack.stream):
        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stack.stream):
            step()
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stack.stream)
        for _ in range(K):
            g.replay()
        e1.record(stack.stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def time_graph(stack: DecodeStack, K: int, W: int):
    """K replays of one captured CUDA graph holding a whole step (L launches)."""
    torch = stack.torch
    with torch.cuda.stream(stack.stream):
        stack.step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stack.stream):
            stack.step()
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stack.stream)
        for _ in range(K):
            g.replay()
        e1.record(stack.stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def sweep(args):
    """34-layer decode stack under a CUDA graph for M in {1,8,16,32,64} and
    FP32 / BF16 state: one JSON line per point (not the bench's main line)."""
    import torch

    from linear_attention_decode_step_gb300 import build, inputs, kda
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, kind = measured_peak()
    Ms = [int(v) for v in args.sweep_m.split(",")]
    for sd in args.sweep_dtypes.split(","):
        for M in Ms:
            stack = DecodeStack(torch, kda, inputs, M, args.layers, sd, args.x_dtype, dev,
                                kernel=args.kernel, columns=args.columns, threads=args.threads,
                                replicate=True)
            K = max(20, min(2000, int(2e5 / M)))
            ms = time_graph(stack, K, args.warmup)
            per_layer_us = ms / K / args.layers * 1e3
            gbs = state_bytes_per_launch(M, sd) / (per_layer_us * 1e-6) / 1e9
            print(json.dumps({"sweep": True, "M": M, "state_dtype": sd, "layers": args.layers,
                              "kernel": args.kernel, "columns": args.columns,
                              "threads": args.threads, "ms_per_stack": ms / K,
                              "us_per_layer": per_layer_us, "state_gbs": gbs,
                              "frac_of_%s_hbm" % kind: gbs / peak}), flush=True)
            del stack
            torch.cuda.empty_cache()


SWEEP_M = (1, 8, 16, 32, 64)
SWEEP_DTYPES = ("f32", "bf16")


def sweep_object(torch, kda, inputs, dev, layers, x_dtype, peak, peak_kind, gpu_id):
    """The 34-layer stack at every M of SWEEP_M with FP32 and BF16 state (one
    CUDA graph of the stack's launches per step, a bounded number of steps per
    point, SM clocks sampled across the sweep). Returns the `sweep` object of
    the bench line."""
    clocks = ClockSampler(gpu_id)
    clocks.start()
    points = []
    for sd in SWEEP_DTYPES:
        for M in SWEEP_M:
            stack = DecodeStack(torch, kda, inputs, M, layers, sd, x_dtype, dev, replicate=True)
            K = max(20, min(300, 3000 // M))
            ms = time_graph(stack, K, 3)
            us = ms / K / layers * 1e3
            gbs = state_bytes_per_launch(M, sd) / (us * 1e-6) / 1e9
            ab = algorithmic_bytes_per_launch(M, sd, x_dtype)
            points.append({"M": M, "state_dtype": sd, "steps": K,
                           "ms_per_stack": ms / K, "us_per_layer": us, "state_gbs": gbs,
                           "state_frac_of_%s_hbm" % peak_kind: gbs / peak,
                           "algorithmic_gbs": ab / (us * 1e-6) / 1e9,
                           "roofline_frac": ab / (us * 1e-6) / 1e9 / peak})
            del stack
            torch.cuda.empty_cache()
    return {"workload": "%d-layer KDA decode stack (one token per step, every layer its own "
                        "state and conv cache, %s q/k/v), M x 64 heads x 128x128 state, for "
                        "M in %s and FP32 / BF16 state storage" % (layers, x_dtype.upper(),
                                                                    list(SWEEP_M)),
            "kernel": DECODE_KERNEL, "launch": "one CUDA graph of %d kda_decode_step launches "
                                                "per step; CUDA events around the replays" % layers,
            "l2": "inputs larger than L2 from M = 8 on (M = 1: 8.4 MB of state per layer, "
                  "285 MB per step for FP32)",
            "points": points, "clocks": clocks.stop()}


def time_e2e(stack: DecodeStack, K: int, W: int, barrier):
    """K steps through the public API with host buffers: every step copies its
    inputs (x, alpha, beta of all layers) in from pinned host memory, runs the
    34 kda_decode_step launches (captured once per buffer set as a CUDA graph)
    and copies o back to pinned host memory. Two buffer sets let the copies of
    neighbouring steps overlap a step's compute (in on one stream, out on
    another); the timed region runs from the first copy in to the last copy
    out."""
    torch = stack.torch
    cs, ds, s = torch.cuda.Stream(), torch.cuda.Stream(), stack.stream
    graphs = []
    with torch.cuda.stream(s):
        for b in range(2):
            stack.step(b)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                stack.step(b)
            graphs.append(g)
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]
    done = [ev(), ev()]
    freed = [ev(), ev()]

    def run(n):
        for k in range(n):
            b = k & 1
            if k >= 2:
                cs.wait_event(freed[b])        # step k-2 is done with buffer set b
            with torch.cuda.stream(cs):
                stack.copy_in(b)
            in_ready[b].record(cs)
            s.wait_event(in_ready[b])
            with torch.cuda.stream(s):   # replay() launches on the current stream
                graphs[b].replay()
            done[b].record(s)
            ds.wait_event(done[b])
            with torch.cuda.stream(ds):
                stack.copy_out(b)
            freed[b].record(ds)

    run(max(3, W))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(cs)
    s.wait_event(e0)
    ds.wait_event(e0)
    run(K)
    ds.wait_event(done[(K - 1) & 1])
    e1.record(ds)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1)


# --------------------------------------------------------------------------- prefill
def prefill_bytes(M, T, H, qkv_bytes=2):
    """Algorithmic bytes of one prefill: q, k, v, alpha, beta in, o out,
    state read and written."""
    tok = M * T * H
    return tok * DH * (3 * qkv_bytes + 4 + 4) + tok * 4 + 2 * M * H * DH * DH * 4


def prefill_flops(M, T, H, chunk=64):
    """Dense contraction flops of the chunked form per (stream, head, chunk),
    counted as the pages count them: two C x C score matrices (2 C^2 d), W and
    U (2 C^2 d), reading and correcting with the state (2 C d^2), the state
    update (C d^2): 2 (4 C^2 d + 3 C d^2) = 2 * 5.24 M at C = 64, d = 128."""
    C = chunk
    macs = 4 * C * C * DH + 3 * C * DH * DH
    return 2 * macs * M * H * ((T + C - 1) // C)


def time_prefill(torch, kda, inputs, M, T, K, W, kernel=0):
    """K chunked prefills of one (M, T, 64-head) problem resident on the GPU,
    timed with CUDA events around the whole run (state updated in place)."""
    p = inputs.prefill_problem(inputs.layer_seed(inputs.SEED_PREFILL_M4_T4096, 0), M=M, T=T, H=H)
    dev = torch.device("cuda")
    bf = lambda bits: torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
    q, k, v = bf(p["q_bits"]), bf(p["k_bits"]), bf(p["v_bits"])
    alpha = torch.from_numpy(p["alpha"]).to(dev)
    beta = torch.from_numpy(p["beta"]).to(dev)
    S = torch.from_numpy(p["S0"]).to(dev)
    o = torch.empty((M, T, H, DH), dtype=torch.float32, device=dev)
    del p
    run = lambda: kda.kda_chunk_prefill_config(q, k, v, alpha, beta, S, o, kernel=kernel)
    for _ in range(W):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        run()
    e1.record()
    torch.cuda.synchronize()
    if kda.kda_device_error() != kda.KDA_OK:
        raise RuntimeError("prefill kernel reported a device-side timeout")
    return e0.elapsed_time(e1) / K


def time_prefill_layer(torch, kda, inputs, M, T, K, W, norm=True):
    """K calls of kda_prefill_layer (conv + gate + chunked recurrence + gated
    RMSNorm) on one (M, T, 64-head) prompt resident on the GPU; state and
    cache updated in place. Returns ms per call."""
    p = inputs.prefill_layer_problem(inputs.layer_seed(inputs.SEED_PREFILL_M4_T4096, 2), M=M, T=T, H=H)
    dev = torch.device("cuda")
    bf = lambda bits: torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
    x, cache = bf(p["x_bits"]), bf(p["cache_bits"])
    t = {n: torch.from_numpy(p[n]).to(dev) for n in ("conv_w", "f", "A_log", "dt_bias", "beta",
                                                   "S0", "out_gate", "norm_w")}
    y = torch.empty((M, T, H, DH), dtype=torch.float32, device=dev)
    del p
    run = lambda: kda.kda_prefill_layer(x, t["conv_w"], cache, t["f"], t["A_log"], t["dt_bias"],
                                        t["beta"], t["S0"], y,
                                        out_gate=t["out_gate"] if norm else None,
                                        norm_weight=t["norm_w"] if norm else None)
    for _ in range(W):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        run()
    e1.record()
    torch.cuda.synchronize()
    if kda.kda_device_error() != kda.KDA_OK:
        raise RuntimeError("prefill layer reported a device-side timeout")
    return e0.elapsed_time(e1) / K


def prefill_layer_bytes(M, T, H, x_bytes=2, norm=True):
    """Algorithmic bytes of one layer prefill: pre-conv x, gate input f, beta
    (and the output gate) in, y out, state and conv cache read and written."""
    tok = M * T * H
    per = 3 * x_bytes + 4 + 4 + (4 if norm else 0)
    return tok * DH * per + tok * 4 + 2 * M * H * DH * DH * 4 + 2 * M * 9 * H * DH * x_bytes


def prefill_summary(ms, M, T, peak_hbm, peak_bf16, kernel_name):
    gb = prefill_bytes(M, T, H) / 1e9
    tflop = prefill_flops(M, T, H) / 1e12
    tf32_peak = peak_bf16 * 1.1 / 2.25   # measured BF16 x the nominal TF32 / BF16 ratio
    return {
        "workload": "chunked prefill, M=%d streams x T=%d tokens x %d heads, 128x128 FP32 state, "
                    "BF16 q/k/v, chunk 64" % (M, T, H),
        "kernel": kernel_name, "ms": ms, "tokens_per_s": M * T / (ms * 1e-3),
        "gb_s": gb / (ms * 1e-3), "frac_of_measured_hbm": gb / (ms * 1e-3) / peak_hbm,
        "algorithmic_bytes": gb * 1e9, "tflop_s": tflop / (ms * 1e-3),
        "frac_of_tf32_peak": tflop / (ms * 1e-3) / tf32_peak,
        "tf32_peak_tflop_s": tf32_peak, "tf32_peak_kind": "measured bf16 x nominal 1.1/2.25",
    }


SM_COUNT = 152          # GB300
FP32_LANES_PER_SM = 128
MAX_SM_MHZ = 2070.0


def fp32_peak_tflops(sm_mhz=None):
    """FP32 FMA peak derived from the unit counts: 152 SMs x 128 lanes x
    2 flop per FMA x the SM clock (the sampled median under load, else the
    2070 MHz maximum)."""
    mhz = sm_mhz if sm_mhz else MAX_SM_MHZ
    return SM_COUNT * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def time_tokens(torch, kda, inputs, M, T, state_dtype, K, W):
    """K multi-token decode calls (T tokens each) of one layer at M streams x
    64 heads, alternating between two state buffers (together larger than L2).
    Returns ms per call."""
    inp = inputs.decode_layer(inputs.layer_seed(inputs.SEED_DECODE_TOKENS, T), M=M, H=H, T=T)
    tok = inputs.stack_tokens(inp)
    dev = torch.device("cuda")
    bf = lambda bits: torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
    x, cache = bf(tok["x_bits"]), bf(inp["cache_bits"])
    w = torch.from_numpy(inp["conv_w"]).to(dev)
    alpha = torch.from_numpy(tok["alpha"]).to(dev)
    beta = torch.from_numpy(tok["beta"]).to(dev)
    S0 = torch.from_numpy(inp["S0"]).to(dev)
    Ss = [S0.to(torch.bfloat16) if state_dtype == "bf16" else S0.clone() for _ in range(2)]
    o = torch.empty((M, T, H, DH), dtype=torch.float32, device=dev)
    del inp, tok
    run = lambda i: kda.kda_decode_tokens(x, w, cache, alpha, beta, Ss[i & 1], o)
    for i in range(W):
        run(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K):
        run(i)
    e1.record()
    torch.cuda.synchronize()
    if kda.kda_device_error() != kda.KDA_OK:
        raise RuntimeError("multi-token decode reported a device-side timeout")
    return e0.elapsed_time(e1) / K


# Calls of at least this many tokens run the chunked multi-token kernel (the
# library's dispatch rule in kda_decode_tokens.cu).
TOKENS_WY_MIN = 3


def tokens_kernel_name(T):
    return "kda_decode_tokens_wy_kernel" if T >= TOKENS_WY_MIN else "kda_decode_tokens_kernel"


def tokens_summary(ms, M, T, state_dtype, peak_hbm, sm_mhz):
    """Roofline of one multi-token call: the state is read and written once
    (HBM), each token costs 7 dk dv flops per head on CUDA cores (fade,
    two column sums, rank-1 correction)."""
    us = ms * 1e3
    sb = state_bytes_per_launch(M, state_dtype)
    flops = 7 * DH * DH * M * H * T
    fp32 = fp32_peak_tflops(sm_mhz)
    t_hbm = sb / (peak_hbm * 1e9) * 1e6
    t_alu = flops / (fp32 * 1e12) * 1e6
    return {"T": T, "us_per_call": us, "us_per_token": us / T,
            "state_gbs": sb / (us * 1e-6) / 1e9,
            "tflop_s": flops / (us * 1e-6) / 1e12,
            "bound": "hbm" if t_hbm >= t_alu else "alu",
            "roofline_us": max(t_hbm, t_alu), "frac_of_roofline": max(t_hbm, t_alu) / us}


def measured_bf16():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


# --------------------------------------------------------------------------- CPU oracle
def oracle_decode_sample(inp, budget_s: float):
    """Times the fp64 oracle's decode step on `inp` until budget_s passes
    (at least one step). Returns (state GB/s, steps, seconds)."""
    import oracle
    M = inp["M"]
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle.decode_step(inp["x_f32"][0], inp["conv_w"], inp["cache_f32"], inp["alpha"][0],
                           inp["beta"][0], inp["S0"])
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return state_bytes_per_launch(M, "f32") * steps / el / 1e9, steps, el


_WORKER_INPUTS = {}
REF_ROUNDS = 20  # oracle pool rounds per reference-arm step


def _oracle_worker(seed: int) -> float:
    """One fp64 oracle decode step of one stream (64 heads) of the layer with
    this seed, in a pool process; returns its seconds."""
    import oracle
    from linear_attention_decode_step_gb300 import inputs
    inp = _WORKER_INPUTS.get(seed)
    if inp is None:
        inp = _WORKER_INPUTS[seed] = inputs.decode_layer(seed, M=1, T=1)
    t0 = time.perf_counter()
    oracle.decode_step(inp["x_f32"][0], inp["conv_w"], inp["cache_f32"], inp["alpha"][0],
                       inp["beta"][0], inp["S0"])
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """The unchanged oracle on every host core: P processes (started with
    spawn, so they never inherit a CUDA context), each decoding its own stream
    (one stream = 64 heads) of a layer. One round = P decode steps at once."""

    def __init__(self, cores: int | None = None):
        import multiprocessing as mp
        import oracle
        oracle.build()  # once, before the workers load it
        self.cores = cores or host_cores()
        self.pool = mp.get_context("spawn").Pool(self.cores)
        self.seeds = [inputs_seed(l) for l in range(self.cores)]
        for _ in range(5):  # workers import, build their inputs, load the oracle, warm up
            self.round()

    def round(self) -> float:
        t0 = time.perf_counter()
        self.pool.map(_oracle_worker, self.seeds, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def inputs_seed(l: int) -> int:
    """Seed of layer l of the 34-layer decode stack."""
    from linear_attention_decode_step_gb300 import inputs
    return inputs.layer_seed(inputs.SEED_DECODE_STACK, l)


def oracle_all_cores_sample(budget_s: float):
    """Rounds of the oracle pool until budget_s passes (at least one).
    Returns (state GB/s, rounds, seconds, cores)."""
    pool = OraclePool()
    rounds, el = 0, 0.0
    while el < budget_s or rounds == 0:
        el += pool.round()
        rounds += 1
    pool.close()
    per_round = state_bytes_per_launch(1, "f32") * pool.cores
    return per_round * rounds / el / 1e9, rounds, el, pool.cores


def config_dict(M, state_dtype, x_dtype, layers=LAYERS):
    return {
        "workload": "KDA decode step, %d-layer stack, M=%d streams x %d heads x %dx%d %s "
                    "state, fused conv+SiLU+L2norm, %s q/k/v and conv cache"
                    % (layers, M, H, DH, DH, state_dtype.upper(), x_dtype.upper()),
        "M": M, "H": H, "dk": DH, "dv": DH, "layers": layers,
        "state_dtype": state_dtype, "x_dtype": x_dtype,
        "l2": "inputs larger than L2: each step touches %d layers x %.0f MB of state, "
              "visited in turn" % (layers, state_bytes_per_launch(M, state_dtype) / 2e6),
        "launch": "one CUDA graph per step holding the %d kda_decode_step launches" % layers,
    }


# --------------------------------------------------------------------------- arms
def reference_arm(args, rank: int):
    """The fp64 CPU oracle on all of this host's cores, on a bounded sample of
    the same workload per step: REF_ROUNDS rounds of one decode step of one
    stream (64 heads) per core, each core on a different layer's inputs."""
    if rank != 0:
        return
    pool = OraclePool()
    for _ in range(args.warmup * REF_ROUNDS):
        pool.round()
    el = 0.0
    for _ in range(args.steps * REF_ROUNDS):
        el += pool.round()
    pool.close()
    per_step_bytes = state_bytes_per_launch(1, "f32") * pool.cores * REF_ROUNDS
    value = per_step_bytes * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(args.M, "f32", "bf16"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.cores, "kind": "oracle",
                         "sample": "per step: %d rounds of one decode step of one stream (64 "
                                   "heads, 128x128 state) on each of %d cores, each on its own "
                                   "layer's inputs, fp64 C oracle, one process per core"
                                   % (REF_ROUNDS, pool.cores)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def own_arm(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    from linear_attention_decode_step_gb300 import build, inputs, kda

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    stack = DecodeStack(torch, kda, inputs, args.M, args.layers, args.state_dtype, args.x_dtype,
                        dev, kernel=args.kernel, columns=args.columns, threads=args.threads,
                        rank=rank)
    clocks = ClockSampler(gpu_uuid(torch, dev))
    clocks.start()
    total_ms, step_ms = time_device(stack, args.steps, args.warmup, barrier)
    clk = clocks.stop()
    e2e_ms = time_e2e(stack, args.steps, max(3, args.warmup // 4), barrier)

    # the job's time is the slowest rank's (the only collective: timing)
    total_ms, e2e_ms = replicas.max_over_ranks([total_ms, e2e_ms], dist if world > 1 else None,
                                               device=dev)

    K = args.steps
    sb = state_bytes_per_launch(args.M, args.state_dtype)
    ab = algorithmic_bytes_per_launch(args.M, args.state_dtype, args.x_dtype)
    L = args.layers
    M_ = args.M
    value = replicas.job_throughput(L * K * sb, world, total_ms * 1e-3) / 1e9
    e2e_value = replicas.job_throughput(L * K * sb, world, e2e_ms * 1e-3) / 1e9
    mean_launch_ms = total_ms / (K * args.layers)   # launch-to-launch, gaps included
    peak, peak_kind = measured_peak()
    achieved = ab / (mean_launch_ms * 1e-3) / 1e9
    traffic = ncu_traffic_per_launch(args.M, args.state_dtype)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if args.state_dtype == "f32" else "f32 (bf16 state storage)",
        "data": "synthetic", "config": config_dict(args.M, args.state_dtype, args.x_dtype),
        "ms_per_layer": total_ms / K / L,
        "ms_per_step_spread": [float(np.min(step_ms)), float(np.median(step_ms)),
                               float(np.max(step_ms))],
        "state_gbs_frac_of_%s_hbm" % peak_kind: value / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": DECODE_KERNEL if args.kernel in (0, 2) else "kda_decode_kernel",
                     "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": ab,
                     "mean_launch_us": mean_launch_ms * 1e3,
                     "launch_timing": "CUDA events around each replay of a graph of %d launches; "
                                      "per launch = step time / %d" % (L, L)},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": stack.h2d_bytes(),
                "d2h_bytes_per_step": stack.d2h_bytes()},
        "gpu_launches": K * L,
        "clocks": clk,
    }
    if not args.no_fused:
        fms = time_fused(stack, inputs, K, 3)
        fus = fms / K / L * 1e3
        fab = ab + M_ * H * DH * 4          # + the output gate read (f replaces alpha)
        line["decode_fused"] = {
            "workload": "the same stack with the forget gate fused in front (raw gate input "
                        "instead of alpha) and the gated RMSNorm fused behind",
            "kernel": "kda_decode_stream_kernel<..., gate, norm>", "us_per_layer": fus,
            "state_gbs": sb / (fus * 1e-6) / 1e9,
            "state_frac_of_%s_hbm" % peak_kind: sb / (fus * 1e-6) / 1e9 / peak,
            "algorithmic_bytes_per_launch": fab,
            "achieved_gbs": fab / (fus * 1e-6) / 1e9}
    if not args.no_prefill:
        pk = {1: "kda_prefill_simt_kernel", 2: "kda_prefill_tc_kernel"}.get(args.prefill_kernel,
                                                                             "kda_prefill_tc_kernel")
        pms = time_prefill(torch, kda, inputs, 4, 4096, min(args.steps, 20), 3,
                           kernel=args.prefill_kernel)
        line["prefill"] = prefill_summary(pms, 4, 4096, peak, measured_bf16(), pk)
        lms = time_prefill_layer(torch, kda, inputs, 4, 4096, min(args.steps, 20), 3)
        lgb = prefill_layer_bytes(4, 4096, H) / 1e9
        line["prefill_layer"] = {
            "workload": "kda_prefill_layer: the same prompt (M=4 x T=4096 x 64 heads) as a whole "
                        "layer: pre-conv BF16 x with the conv cache, raw gate input, chunked "
                        "recurrence, gated RMSNorm",
            "kernel": "kda_prefill_tc_kernel<bf16, layer, norm>", "ms": lms,
            "tokens_per_s": 4 * 4096 / (lms * 1e-3), "gb_s": lgb / (lms * 1e-3),
            "frac_of_measured_hbm": lgb / (lms * 1e-3) / peak,
            "algorithmic_bytes": lgb * 1e9}
    if not args.no_tokens:
        mhz = clk.get("sm_mhz") if isinstance(clk, dict) else None
        rows = [tokens_summary(time_tokens(torch, kda, inputs, M_, T, args.state_dtype, 30, 3),
                               M_, T, args.state_dtype, peak, mhz) for T in (2, 4, 8, 16)]
        for r in rows:
            r["kernel"] = tokens_kernel_name(r["T"])
        line["decode_tokens"] = {
            "workload": "multi-token decode (kda_decode_tokens): one layer, M=%d streams x 64 "
                        "heads, T tokens per call, %s state, BF16 q/k/v" % (M_, args.state_dtype),
            "kernel": "kda_decode_tokens_kernel (T < %d), kda_decode_tokens_wy_kernel (T >= %d)"
                      % (TOKENS_WY_MIN, TOKENS_WY_MIN),
            "fp32_peak_tflop_s": fp32_peak_tflops(mhz),
            "fp32_peak_kind": "152 SMs x 128 FP32 lanes x 2 x SM clock (%s MHz)"
                              % ("sampled %.0f" % mhz if mhz else "max 2070"),
            "per_T": rows}
    if not args.no_sweep:
        line["sweep"] = sweep_object(torch, kda, inputs, dev, args.layers, args.x_dtype, peak,
                                     peak_kind, gpu_uuid(torch, dev))
    if world == 1 and not args.no_cpu_baseline:
        gbs1, n1, el1 = oracle_decode_sample(stack.host0, args.cpu_seconds / 3)
        gbs, n, el, cores = oracle_all_cores_sample(2 * args.cpu_seconds / 3)
        line["cpu_baseline"] = {
            "value": gbs, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d rounds in %.1f s of one fp64 C oracle decode step on each of %d "
                      "cores, each core on one stream (64 heads, 128x128 state) of its own "
                      "layer; one process per core" % (n, el, cores),
            "single_thread": {"value": gbs1, "cores": 1,
                              "sample": "layer 0 of the workload (M=%d) decoded %d times, "
                                        "%.1f s" % (args.M, n1, el1)}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--M", type=int, default=32)
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="layers in the stack (34 in GLM-5.3-Flash; fewer only for profiling)")
    ap.add_argument("--state-dtype", choices=["f32", "bf16"], default="f32")
    ap.add_argument("--x-dtype", choices=["f32", "bf16"], default="bf16")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--kernel", type=int, default=0,
                    help="0 auto, 1 cluster (with --columns/--threads), 2 persistent stream")
    ap.add_argument("--columns", type=int, default=0)
    ap.add_argument("--threads", type=int, default=0)
    ap.add_argument("--no-fused", action="store_true",
                    help="skip the decode step with the gate and the gated norm fused in")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the chunked-prefill measurement")
    ap.add_argument("--prefill-kernel", type=int, default=0, help="0 auto, 1 SIMT, 2 tensor core")
    ap.add_argument("--no-tokens", action="store_true",
                    help="skip the multi-token decode leg")
    ap.add_argument("--tokens-only", action="store_true",
                    help="time only kda_decode_tokens at --M streams and --tokens-T tokens")
    ap.add_argument("--tokens-T", type=int, default=4)
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prefill (with --prefill-M/--prefill-T), one JSON line")
    ap.add_argument("--prefill-layer", action="store_true",
                    help="with --prefill-only: time kda_prefill_layer instead")
    ap.add_argument("--prefill-M", type=int, default=4)
    ap.add_argument("--prefill-T", type=int, default=4096)
    ap.add_argument("--sweep", action="store_true",
                    help="time the 34-layer stack for several M and state dtypes instead")
    ap.add_argument("--sweep-m", default="1,8,16,32,64")
    ap.add_argument("--sweep-dtypes", default="f32,bf16")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the sweep object (the stack at M = 1..64, FP32 and BF16 state)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    if args.sweep:
        sweep(args)
        return
    if args.tokens_only:
        import torch
        from linear_attention_decode_step_gb300 import build, inputs, kda
        build.build()
        ms = time_tokens(torch, kda, inputs, args.M, args.tokens_T, args.state_dtype, args.steps,
                         args.warmup)
        print(json.dumps(tokens_summary(ms, args.M, args.tokens_T, args.state_dtype,
                                        measured_peak()[0], None)))
        return
    if args.prefill_only:
        import torch
        from linear_attention_decode_step_gb300 import build, inputs, kda
        build.build()
        torch.cuda.set_device(0)
        peak, _ = measured_peak()
        if args.prefill_layer:
            lms = time_prefill_layer(torch, kda, inputs, args.prefill_M, args.prefill_T,
                                     args.steps, args.warmup)
            lgb = prefill_layer_bytes(args.prefill_M, args.prefill_T, H) / 1e9
            print(json.dumps({"kernel": "kda_prefill_layer", "M": args.prefill_M,
                              "T": args.prefill_T, "ms": lms,
                              "tokens_per_s": args.prefill_M * args.prefill_T / (lms * 1e-3),
                              "frac_of_measured_hbm": lgb / (lms * 1e-3) / peak}))
            return
        pms = time_prefill(torch, kda, inputs, args.prefill_M, args.prefill_T, args.steps,
                           args.warmup, kernel=args.prefill_kernel)
        print(json.dumps(prefill_summary(pms, args.prefill_M, args.prefill_T, peak,
                                         measured_bf16(), "kernel %d" % args.prefill_kernel)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        own_arm(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
