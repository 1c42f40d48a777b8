#!/usr/bin/env python
"""Benchmark of the selective scan (S6) and its decode state update on B300.

One step = one selective-scan pass (softplus step, discretisation, recurrence,
readout, gate, final state) over the Mamba-130M-layer workload: batch 8,
d_inner 1536, L 2048, N 16, bf16 io with fp32 state. The metric is
element-steps per second (batch * d_inner * L * N / s), with achieved HBM GB/s
as a fraction of the measured copy bandwidth in the roofline object.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch with torch.distributed.run; every rank scans its own batch
shard (independent sequences, no collective on the data path: weak scaling).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_138_b300 import inputs as I  # noqa: E402

HEADLINE = I.MAMBA130M
METRIC = "selective-scan element-steps/s (B*D*L*N)"
UNIT = "element-steps/s"
L2_FLUSH_BYTES = 256 << 20  # > the 126 MB L2
# A device-side wait enqueued after the flush and before each start event of a
# short kernel (the conv kernels, the tiny scan), so that the host has enqueued
# the timed launch before the event fires: the measured interval then holds the
# kernel, not the host's launch latency. Long kernels need no cover.
LAUNCH_COVER_CYCLES = 2_000_000   # about 1 ms at the B300 clock
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
SRC = os.path.join(ROOT, "selective_state_space_138_b300", "csrc", "ss_scan.cu")


# ----------------------------------------------------------------- helpers

def io_bytes(io: str) -> int:
    return 2 if io == "bf16" else 4


def scan_alg_bytes(spec: I.ScanSpec, final_state: bool = True) -> int:
    """Bytes the fused scan must move: read x, dt, z and write y (batch, d_inner,
    L); read B, C (batch, N, L); read A (d_inner, N), D and dt_bias; write the
    final state (batch, d_inner, N) fp32."""
    s = io_bytes(spec.io)
    bdl = spec.batch * spec.d_inner * spec.L
    b = 4 * bdl * s + spec.batch * spec.L * 2 * spec.N * s + spec.d_inner * spec.N * 4 + 2 * spec.d_inner * 4
    if final_state:
        b += spec.batch * spec.d_inner * spec.N * 4
    return b


def bwd_alg_bytes(spec: I.ScanSpec) -> int:
    """Bytes the backward pass must move: read x, dt, z, dout and write dx,
    ddelta, dz (batch, d_inner, L); read B, C (batch, N, L) and write dB, dC in
    fp32; read A, D, dt_bias and write dA, dD, ddt_bias. The states it
    recomputes are not counted (they are never stored in full)."""
    s = io_bytes(spec.io)
    bdl = spec.batch * spec.d_inner * spec.L
    bnl = spec.batch * spec.N * spec.L
    return 7 * bdl * s + bnl * 2 * s + bnl * 2 * 4 + 2 * spec.d_inner * spec.N * 4 + 4 * spec.d_inner * 4


def decode_alg_bytes(spec: I.DecodeSpec) -> int:
    """Per step: read and write the fp32 state, read x, delta, z and write y,
    read B, C, A and D."""
    bd = spec.batch * spec.d_inner
    return 2 * bd * spec.N * 4 + 4 * bd * 2 + 2 * spec.batch * spec.N * 2 + spec.d_inner * spec.N * 4 + spec.d_inner * 4


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count \
        if torch.cuda.is_available() else 148
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured", "sms": sms,
                "sm_max_mhz": float(d.get("sm_max_mhz", 2032.0)),
                "bf16_tflops": float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS))}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback", "sms": sms, "sm_max_mhz": 2032.0,
                "bf16_tflops": FALLBACK_BF16_TFLOPS}


# the source part each profiled kernel lives in (besides the shared device helpers)
KERNEL_PART = {"scan_fwd_": ("scan_fwd.cuh",), "state_update_": ("decode.cuh",),
               "scan_bwd_": ("scan_bwd.cuh",), "conv1d_": ("conv.cuh",), "conv_state_update_": ("conv.cuh",),
               "ssd_chunk_": ("ssd.cuh",)}


def kernel_source_hash(kernel_key: str) -> str:
    """sha256 of the shared device helpers followed by the kernel's own files."""
    parts = next(v for k, v in KERNEL_PART.items() if kernel_key.startswith(k))
    csrc = os.path.dirname(SRC)
    h = hashlib.sha256()
    for name in ("device_common.cuh", *parts):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()


def profiled_traffic(kernel_key: str):
    """Bytes per launch (dram read + write) from the committed ncu summary of
    ``kernel_key``, when the kernel's source has not changed since the capture
    (``source_sha256`` as computed by ``kernel_source_hash``)."""
    src_hash = kernel_source_hash(kernel_key)
    path = os.path.join(ROOT, "profiles", kernel_key + ".md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        item = line.strip().lstrip("-").strip().strip("`")   # "- `key: value`"
        if ":" in item and item.startswith(("traffic_bytes_per_launch", "source_sha256")):
            k, v = item.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256") != src_hash:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class L2Flush:
    """Run between timed launches: write a buffer larger than L2 (its lines
    replace whatever the previous launch left there), then read a second one
    of the same size, so that the write's dirty lines are written back to DRAM
    here, before the timed launch, and not while it runs."""

    def __init__(self):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.out = torch.empty(1, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r.view(1, -1), dim=1, out=self.out)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        busy = [s for s, p in zip(sm, power)]
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm),
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def reduce_max(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- GPU arm

def shard_spec(spec: I.ScanSpec, rank: int) -> I.ScanSpec:
    """Rank r scans its own batch shard: the same shape, a distinct seed."""
    import dataclasses
    return dataclasses.replace(spec, seed=spec.seed + 1000 * rank)


def time_scan(spec: I.ScanSpec, steps: int, warmup: int, flush: bool = True, soak_s: float = 0.0,
              cover: bool = False):
    """Per-launch device times (ms) of the scan kernel over ``steps`` launches,
    each preceded by an L2 flush; events on the launching stream. ``cover``
    adds the device-side wait before each start event, so that the host's work
    for the call (argument checks, tensor-map encoding, the launch) is done
    before the start event fires and no idle gap enters the measurement."""
    from selective_state_space_138_b300 import binding
    inp = I.make_scan_inputs(spec)
    g = {k: v.cuda() for k, v in inp.items() if k != "reset_pos"}
    y = torch.empty_like(g["x"])
    fs = torch.empty(spec.batch, spec.d_inner, spec.N, device="cuda", dtype=torch.float32)
    scratch = L2Flush()

    def run():
        binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"],
                         y=y, final_state=fs)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    if soak_s > 0:  # untimed: let clocks settle under this load
        t_end = time.time() + soak_s
        while time.time() < t_end:
            for _ in range(20):
                run()
            torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        if flush:
            scratch()
        if cover:
            torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        starts[i].record()
        run()
        ends[i].record()
    torch.cuda.synchronize()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    del g, y, fs, scratch
    torch.cuda.empty_cache()
    return times


def time_scan_e2e(spec: I.ScanSpec, steps: int, warmup: int):
    """Same metric through the C ABI with pinned host buffers: every step copies
    its inputs host->device, scans, and copies y and the final state back.
    Steps are pipelined over three streams with two buffer sets, as a serving
    loop would run them: step k's inputs travel while step k-1 is scanned and
    step k-2's outputs come back (each copy engine and the SMs stay busy).
    Returns (ms per step, H2D bytes per step, D2H bytes per step)."""
    from selective_state_space_138_b300 import binding
    inp = I.make_scan_inputs(spec)
    keys = ("x", "dt", "z", "B", "C", "A", "D", "dt_bias")
    host = {k: inp[k].pin_memory() for k in keys}
    sets = []
    for _ in range(2):
        g = {k: torch.empty_like(host[k], device="cuda") for k in keys}
        y = torch.empty_like(g["x"])
        fs = torch.empty(spec.batch, spec.d_inner, spec.N, device="cuda", dtype=torch.float32)
        y_h = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        fs_h = torch.empty(fs.shape, dtype=fs.dtype, pin_memory=True)
        sets.append(dict(g=g, y=y, fs=fs, y_h=y_h, fs_h=fs_h, ev_in=torch.cuda.Event(), ev_comp=torch.cuda.Event(),
                         ev_out=torch.cuda.Event(), used=False))
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sets[0]["y"].numel() * sets[0]["y"].element_size() + sets[0]["fs"].numel() * 4
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def step(k):
        st = sets[k % 2]
        with torch.cuda.stream(s_in):
            if st["used"]:
                s_in.wait_event(st["ev_comp"])        # the scan that read this set is done
            for key in keys:
                st["g"][key].copy_(host[key], non_blocking=True)
            st["ev_in"].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(st["ev_in"])
            if st["used"]:
                s_comp.wait_event(st["ev_out"])       # this set's previous outputs have been read back
            g = st["g"]
            binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"],
                             y=st["y"], final_state=st["fs"], stream=s_comp)
            st["ev_comp"].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(st["ev_comp"])
            st["y_h"].copy_(st["y"], non_blocking=True)
            st["fs_h"].copy_(st["fs"], non_blocking=True)
            st["ev_out"].record(s_out)
        st["used"] = True

    for k in range(warmup):
        step(k)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for k in range(warmup, warmup + steps):
        step(k)
    s_in.wait_stream(s_out)
    end.record(s_in)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, h2d, d2h


def time_decode(spec: I.DecodeSpec, reps: int, warmup: int):
    """1024 consecutive single-token updates captured in one CUDA graph; also
    the same updates launched one by one with an L2 flush before each."""
    from selective_state_space_138_b300 import binding
    tok = I.make_decode_tokens(spec)
    par = I.make_decode_params(spec)
    gt = {k: v.cuda() for k, v in tok.items()}
    del tok
    A = par["A"].cuda()
    D = par["D"].cuda()
    state = torch.zeros(spec.batch, spec.d_inner, spec.N, device="cuda")
    ys = torch.empty_like(gt["x"])
    T = spec.steps

    def chain():
        for t in range(T):
            binding.state_update(state, gt["x"][t], gt["delta"][t], A, gt["B"][t], gt["C"][t], D=D, z=gt["z"][t],
                                 y=ys[t])

    chain()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
            chain()
    torch.cuda.synchronize()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(reps):
        graph.replay()
    ev[1].record()
    torch.cuda.synchronize()
    graph_ms_per_token = ev[0].elapsed_time(ev[1]) / (reps * T)

    scratch = L2Flush()
    n_flushed = min(T, 64)
    st = [torch.cuda.Event(enable_timing=True) for _ in range(n_flushed)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(n_flushed)]
    for t in range(n_flushed):
        scratch()
        torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        st[t].record()
        binding.state_update(state, gt["x"][t], gt["delta"][t], A, gt["B"][t], gt["C"][t], D=D, z=gt["z"][t],
                             y=ys[t])
        en[t].record()
    torch.cuda.synchronize()
    flushed_ms = statistics.median([a.elapsed_time(b) for a, b in zip(st, en)])
    del gt, ys, state, scratch, graph
    torch.cuda.empty_cache()
    return graph_ms_per_token, flushed_ms


def time_conv(spec: I.ScanSpec, steps: int, warmup: int, k: int = 4):
    """Causal conv1d + SiLU over the layer input, L2 flushed before each launch.
    Returns (median ms, algorithmic bytes: x read, out written, weights, bias,
    history written)."""
    from selective_state_space_138_b300 import binding
    x = I.normal(spec.seed, 11, (spec.batch, spec.d_inner, spec.L), 1.0, torch.bfloat16).cuda()
    w = I.normal(spec.seed, 12, (spec.d_inner, k), 0.5, torch.float32).cuda()
    bias = I.normal(spec.seed, 13, (spec.d_inner,), 0.2, torch.float32).cuda()
    out = torch.empty_like(x)
    st = torch.empty((spec.batch, k - 1, spec.d_inner), dtype=x.dtype, device="cuda")
    scratch = L2Flush()
    for _ in range(warmup):
        binding.causal_conv1d(x, w, bias, out=out, state_out=st)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        scratch()
        torch.cuda._sleep(LAUNCH_COVER_CYCLES)
        a.record()
        binding.causal_conv1d(x, w, bias, out=out, state_out=st)
        b.record()
    torch.cuda.synchronize()
    ms = statistics.median([a.elapsed_time(b) for a, b in ev])
    bdl = spec.batch * spec.d_inner * spec.L
    return ms, 2 * bdl * 2 + spec.d_inner * (k + 1) * 4 + spec.batch * (k - 1) * spec.d_inner * 2


def time_conv_step(spec: I.DecodeSpec, steps: int, k: int = 4):
    """One decode step of the convolution on the decode workload's shape, L2
    flushed before each launch. Returns (median ms, algorithmic bytes, median
    ms of a plain device copy that moves the same bytes under the same
    protocol: the floor a launch of this size meets)."""
    from selective_state_space_138_b300 import binding
    x = I.normal(spec.seed, 11, (spec.batch, spec.d_inner), 1.0, torch.bfloat16).cuda()
    w = I.normal(spec.seed, 12, (spec.d_inner, k), 0.5, torch.float32).cuda()
    bias = I.normal(spec.seed, 13, (spec.d_inner,), 0.2, torch.float32).cuda()
    st = I.normal(spec.seed, 14, (spec.batch, k - 1, spec.d_inner), 1.0, torch.bfloat16).cuda()
    out = torch.empty_like(x)
    bd = spec.batch * spec.d_inner
    nbytes = bd * 2 * 2 + 2 * bd * (k - 1) * 2 + spec.d_inner * (k + 1) * 4
    src = torch.zeros(nbytes // 4, dtype=torch.float32, device="cuda")
    dst = torch.empty_like(src)
    scratch = L2Flush()

    def timed(fn):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            scratch()
            torch.cuda._sleep(LAUNCH_COVER_CYCLES)
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median([a.elapsed_time(b) for a, b in ev])

    ms = timed(lambda: binding.conv_state_update(st, x, w, bias, out=out))
    copy_ms = timed(lambda: dst.copy_(src))
    return ms, nbytes, copy_ms


def time_bwd(spec: I.ScanSpec, steps: int, warmup: int, from_forward: bool = False, variant: bool = False):
    """Median device time (ms) of the backward pass over ``steps`` launches,
    each preceded by an L2 flush; outputs and workspace preallocated. With
    ``from_forward`` the workspace is filled once by the training forward and
    every timed backward skips its own forward walk; the training forward's
    median time is then returned too. With ``variant`` the gradient of the
    reverse-direction scan with a sequence start every 250 steps is timed
    instead."""
    from selective_state_space_138_b300 import binding
    inp = I.make_scan_inputs(spec)
    g = {k: inp[k].cuda() for k in ("x", "dt", "z", "B", "C", "A", "D", "dt_bias")}
    dout = I.make_bwd_inputs(spec)["dout"].cuda()
    ws = torch.empty(binding.scan_bwd_workspace_bytes(spec.batch, spec.d_inner, spec.L, spec.N),
                     dtype=torch.uint8, device="cuda")
    scratch = L2Flush()
    grads = None
    starts = None
    if variant:
        starts = torch.zeros(spec.batch, spec.L, dtype=torch.uint8)
        starts[:, ::250] = 1
        starts = starts.cuda()

    def run():
        if variant:
            return binding.scan_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, D=g["D"], z=g["z"],
                                    dt_bias=g["dt_bias"], grads=grads, workspace=ws, seq_start=starts, reverse=True)
        return binding.scan_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, D=g["D"], z=g["z"],
                                dt_bias=g["dt_bias"], grads=grads, workspace=ws, states_from_forward=from_forward)

    fwd_ms = None
    if from_forward:
        y = torch.empty_like(g["x"])
        fs = torch.empty(spec.batch, spec.d_inner, spec.N, device="cuda", dtype=torch.float32)
        fwd = lambda: binding.scan_fwd_train(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                             dt_bias=g["dt_bias"], y=y, final_state=fs, workspace=ws)
        for _ in range(warmup):
            fwd()
        fe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in fe:
            scratch()
            torch.cuda._sleep(LAUNCH_COVER_CYCLES)   # the launch is queued before the start event fires
            a.record()
            fwd()
            b.record()
        torch.cuda.synchronize()
        fwd_ms = statistics.median([a.elapsed_time(b) for a, b in fe])
    grads = run()
    for _ in range(warmup):
        run()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        scratch()
        a.record()
        run()
        b.record()
    torch.cuda.synchronize()
    ms = statistics.median([a.elapsed_time(b) for a, b in ev])
    return (ms, fwd_ms) if from_forward else ms


def ssd_alg(spec: I.SsdSpec):
    """(bytes, flops) the scalar-decay scan must move and compute: read x, z,
    dt and write y (batch, L, H, P / H); read B, C (batch, L, G, N); A, D,
    dt_bias; write the final state (batch, H, P, N) fp32. FLOPs: the chunked
    algorithm's products, 2 Q^2 N per (batch, chunk, group) for C B^T and
    2 Q^2 P + 4 Q N P per (batch, chunk, head) for the masked product, the
    state readout and the state update (Q = 64)."""
    b, L, H, P, G, N = spec.batch, spec.L, spec.nheads, spec.headdim, spec.ngroups, spec.N
    q = 64
    chunks = (L + q - 1) // q
    by = 3 * b * L * H * P * 2 + b * L * H * 2 + 2 * b * L * G * N * 2 + 3 * H * 4 + b * H * P * N * 4
    fl = b * chunks * (G * 2 * q * q * N + H * (2 * q * q * P + 4 * q * N * P))
    return by, fl


def time_ssd(spec: I.SsdSpec, steps: int, warmup: int):
    """Median device time (ms) of the scalar-decay scan (both kernels), L2
    flushed before each launch."""
    from selective_state_space_138_b300 import binding
    inp = I.make_ssd_inputs(spec)
    g = {k: v.cuda() for k, v in inp.items()}
    y = torch.empty_like(g["x"])
    fs = torch.empty(spec.batch, spec.nheads, spec.headdim, spec.N, device="cuda")
    ws = torch.empty(binding.ssd_workspace_bytes(spec.batch, spec.L, spec.nheads, spec.ngroups, spec.N), dtype=torch.uint8, device="cuda")
    scratch = L2Flush()

    def run():
        binding.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"], y=y,
                        final_state=fs, workspace=ws)

    for _ in range(warmup):
        run()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        scratch()
        a.record()
        run()
        b.record()
    torch.cuda.synchronize()
    return statistics.median([a.elapsed_time(b) for a, b in ev])


def roofline_obj(alg_bytes: float, ms: float, peaks: dict, traffic, elem_steps: float | None = None):
    """HBM roofline of one launch: algorithmic bytes / launch time against the
    measured copy bandwidth. For a scan, also the fraction of the ALU ceiling:
    one exponential (MUFU ex2, 32 per clock per SM) and four FMA-pipe
    operations (128 lanes per clock per SM) per element-step, i.e. 32
    element-steps per clock per SM at the maximum SM clock."""
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    out = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
           "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured"
           else "fallback 6400 GB/s"}
    if elem_steps is not None:
        ceiling = peaks["sms"] * 32 * peaks["sm_max_mhz"] * 1e6
        rate = elem_steps / (ms * 1e-3)
        out["alu_ceiling"] = {"elem_steps_per_s": ceiling, "achieved": rate, "frac": round(rate / ceiling, 4),
                              "derivation": "%d SMs x 32 element-steps/clk x %.0f MHz" % (peaks["sms"], peaks["sm_max_mhz"])}
        out["floors_us"] = scan_floors_us(alg_bytes, elem_steps, peaks)
    return out


def scan_floors_us(alg_bytes: float, elem_steps: float, peaks: dict) -> dict:
    """The three lower bounds on a scan launch (microseconds): HBM (algorithmic
    bytes at the measured copy bandwidth), the exponentials (one MUFU ex2 per
    element-step, 32 per clock per SM) and fp32 issue (four FMA-pipe
    operations per element-step, packed two to an f32x2 instruction, 128
    lanes per clock per SM), at the maximum SM clock."""
    clk = peaks["sm_max_mhz"] * 1e6
    return {"hbm": round(alg_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6, 2),
            "exp": round(elem_steps / (peaks["sms"] * 32 * clk) * 1e6, 2),
            "fp32_issue": round(elem_steps * 4 / (peaks["sms"] * 128 * 2 * clk) * 1e6, 2)}


# ----------------------------------------------------------------- CPU (oracle)

def oracle_rate(spec: I.ScanSpec, budget_s: float, inp=None):
    """The float64 oracle timed on this host's cores on a bounded sample of the
    workload's rows (whole rows, every time step): the sample grows until one
    timed pass over it takes about budget_s; when the whole workload takes less
    than that, whole passes over it are repeated (at most 20). Returns
    (elem-steps/s, cores, sample description, seconds of the timed passes)."""
    from oracle import oracle as O
    inp = inp if inp is not None else I.make_scan_inputs(spec)
    cores = O.default_threads()
    rows_total = spec.batch * spec.d_inner
    O.scan_rows(inp, list(range(min(rows_total, cores))), threads=cores)   # first call: library load, page faults

    def sample(n):
        stride = max(1, rows_total // n)
        return list(range(0, rows_total, stride))[:n], stride

    n = min(rows_total, 4 * cores)
    while True:
        rows, stride = sample(n)
        t = time.time()
        O.scan_rows(inp, rows, threads=cores)
        sec = time.time() - t
        if sec >= 0.5 * budget_s or n >= rows_total:
            break
        n = min(rows_total, max(2 * n, int(n * 0.9 * budget_s / max(sec, 1e-3))))
    passes = 1
    while len(rows) == rows_total and sec < budget_s and passes < 20:
        t = time.time()
        O.scan_rows(inp, rows, threads=cores)
        sec += time.time() - t
        passes += 1
    elems = passes * len(rows) * spec.L * spec.N
    desc = "%d of %d (batch, channel) rows, every %d-th, all %d steps x %d states" % (
        len(rows), rows_total, stride, spec.L, spec.N)
    if passes > 1:
        desc += ", %d passes" % passes
    return elems / sec, cores, desc, sec


def oracle_single_thread_rate(spec: I.ScanSpec, rows: int = 16, inp=None):
    """The float64 oracle on one host thread over the workload's first rows
    (elem-steps/s)."""
    from oracle import oracle as O
    inp = inp if inp is not None else I.make_scan_inputs(spec)
    O.scan_rows(inp, [0], threads=1)
    t = time.time()
    O.scan_rows(inp, list(range(rows)), threads=1)
    return rows * spec.L * spec.N / (time.time() - t)


def bench_config(spec: I.ScanSpec, world: int) -> dict:
    """The ``config`` object of both arms' lines (the same keys and values, so
    that the two lines describe the same workload)."""
    return {"workload": spec.name, "batch": spec.batch, "d_inner": spec.d_inner, "L": spec.L, "N": spec.N,
            "io": spec.io, "per_gpu": True,
            "l2": "GPU arm: flushed before every step (256 MB written, then 256 MB read, so the write-back of the "
                  "written lines happens before the step)",
            "parallelism": "dp%d (independent batch shards)" % world}


def reference_arm(args, rank, world):
    """The oracle as the reference arm: rank 0 only, host cores."""
    if rank != 0:
        return 0
    spec = HEADLINE
    inp = I.make_scan_inputs(spec)
    for _ in range(args.warmup):
        oracle_rate(spec, budget_s=1.0, inp=inp)
    rates, secs = [], 0.0
    desc, cores = "", 1
    t0 = time.time()
    for _ in range(args.steps):
        r, cores, desc, s = oracle_rate(spec, budget_s=2.0, inp=inp)
        rates.append(r)
        secs += s
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(spec, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(time.time() - t0, 2),
    }
    print(json.dumps(line), flush=True)
    return 0


def ncu_case(args):
    """Launches of one kernel only (for ncu): ``warmup + steps`` launches of the
    headline scan on the same inputs, or of the decode update on the first
    ``warmup + steps`` tokens of the decode workload; no L2 flush, no other
    kernels of this library."""
    from selective_state_space_138_b300 import binding
    torch.cuda.set_device(0)
    if args.ncu_case == "decode":
        spec = I.DECODE
        T = args.warmup + args.steps
        tok = {k: v.cuda() for k, v in I.make_decode_tokens(spec, steps=T).items()}
        par = I.make_decode_params(spec)
        A, Dp = par["A"].cuda(), par["D"].cuda()
        state = torch.zeros(spec.batch, spec.d_inner, spec.N, device="cuda")
        y = torch.empty_like(tok["x"])
        for t in range(T):
            binding.state_update(state, tok["x"][t], tok["delta"][t], A, tok["B"][t], tok["C"][t], D=Dp,
                                 z=tok["z"][t], y=y[t])
        torch.cuda.synchronize()
        return 0
    if args.ncu_case in ("bwd", "bwd_rev", "bwd_longseq_l16384"):
        # bwd_longseq_l16384: the long-sequence rows cut to L = 16384 (an eighth), small
        # enough for a full capture; the long sequence's traffic is 8 times its own
        spec = {"bwd": HEADLINE, "bwd_rev": HEADLINE,
                "bwd_longseq_l16384": dataclasses.replace(I.LONGSEQ, L=I.LONGSEQ.L // 8)}[args.ncu_case]
        inp = I.make_scan_inputs(spec)
        g = {k: v.cuda() for k, v in inp.items() if k != "reset_pos"}
        dout = I.make_bwd_inputs(spec)["dout"].cuda()
        starts = None
        if args.ncu_case == "bwd_rev":   # as the bench's variant line: reversed, a start every 250 steps
            starts = torch.zeros(spec.batch, spec.L, dtype=torch.uint8)
            starts[:, ::250] = 1
            starts = starts.cuda()
        grads = None
        for _ in range(args.warmup + args.steps):
            if starts is not None:
                grads = binding.scan_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, D=g["D"], z=g["z"],
                                         dt_bias=g["dt_bias"], grads=grads, seq_start=starts, reverse=True)
            else:
                grads = binding.scan_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, D=g["D"], z=g["z"],
                                         dt_bias=g["dt_bias"], grads=grads)
        torch.cuda.synchronize()
        return 0
    if args.ncu_case == "ssd":
        spec = I.MAMBA2_LAYER
        inp = I.make_ssd_inputs(spec)
        g = {k: v.cuda() for k, v in inp.items()}
        ws = torch.empty(binding.ssd_workspace_bytes(spec.batch, spec.L, spec.nheads, spec.ngroups, spec.N), dtype=torch.uint8,
                         device="cuda")
        for _ in range(args.warmup + args.steps):
            binding.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"],
                            workspace=ws)
        torch.cuda.synchronize()
        return 0
    if args.ncu_case == "conv":
        spec, k = HEADLINE, 4
        x = I.normal(spec.seed, 11, (spec.batch, spec.d_inner, spec.L), 1.0, torch.bfloat16).cuda()
        w = I.normal(spec.seed, 12, (spec.d_inner, k), 0.5, torch.float32).cuda()
        bias = I.normal(spec.seed, 13, (spec.d_inner,), 0.2, torch.float32).cuda()
        out = torch.empty_like(x)
        st = torch.empty((spec.batch, k - 1, spec.d_inner), dtype=x.dtype, device="cuda")
        for _ in range(args.warmup + args.steps):
            binding.causal_conv1d(x, w, bias, out=out, state_out=st)
        torch.cuda.synchronize()
        return 0
    if args.ncu_case == "conv_step":
        spec, k = I.DECODE, 4
        x = I.normal(spec.seed, 11, (spec.batch, spec.d_inner), 1.0, torch.bfloat16).cuda()
        w = I.normal(spec.seed, 12, (spec.d_inner, k), 0.5, torch.float32).cuda()
        bias = I.normal(spec.seed, 13, (spec.d_inner,), 0.2, torch.float32).cuda()
        st = I.normal(spec.seed, 14, (spec.batch, k - 1, spec.d_inner), 1.0, torch.bfloat16).cuda()
        out = torch.empty_like(x)
        for _ in range(args.warmup + args.steps):
            binding.conv_state_update(st, x, w, bias, out=out)
        torch.cuda.synchronize()
        return 0
    spec = {"scan_1p4b": I.MAMBA1P4B, "scan_longseq": I.LONGSEQ}.get(args.ncu_case, HEADLINE)
    inp = I.make_scan_inputs(spec)
    g = {k: v.cuda() for k, v in inp.items() if k != "reset_pos"}
    y = torch.empty_like(g["x"])
    fs = torch.empty(spec.batch, spec.d_inner, spec.N, device="cuda", dtype=torch.float32)
    for _ in range(args.warmup + args.steps):
        binding.scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"], dt_bias=g["dt_bias"],
                         y=y, final_state=fs)
    torch.cuda.synchronize()
    return 0


# ----------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--headline-only", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-soak", action="store_true", help="skip the 1 s untimed soak before timing")
    ap.add_argument("--ncu-case", choices=["scan", "scan_1p4b", "scan_longseq", "decode", "conv", "conv_step", "bwd",
                                           "bwd_rev", "bwd_longseq_l16384", "ssd"],
                    default=None,
                    help="profiling case: warmup + steps launches of one kernel on its workload (the headline "
                         "scan, the 1.4B-layer or long-sequence scan, the decode update on the first warmup + "
                         "steps tokens, conv, backward, SSD), nothing else")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank, world, local = dist_env()
    if args.ncu_case:
        return ncu_case(args)
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    gpu_index = torch.cuda.current_device()

    from selective_state_space_138_b300 import binding
    binding.lib()  # fails loudly if the CUDA library is missing

    peaks = measured_peaks()
    spec = shard_spec(HEADLINE, rank)

    sampler = ClockSampler(gpu_index) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.time()
    times = time_scan(spec, args.steps, args.warmup, flush=True, soak_s=0.0 if args.no_soak else 1.0, cover=True)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.time() - t_wall
    clocks = sampler.stop() if sampler else None

    total_ms = sum(times)
    total_ms_max = reduce_max(total_ms, world)
    ms_per_step = total_ms_max / args.steps
    elems = spec.elem_steps
    value = world * elems / (ms_per_step * 1e-3)
    alg = scan_alg_bytes(spec)
    traffic = profiled_traffic("scan_fwd_" + HEADLINE.name)

    e2e_ms, h2d, d2h = time_scan_e2e(spec, max(8, args.steps // 2), 3)
    e2e_ms = reduce_max(e2e_ms, world)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
        "config": bench_config(HEADLINE, world),
        "kernel_ms": {"median": statistics.median(times), "min": min(times), "max": max(times)},
        "roofline": roofline_obj(alg, ms_per_step, peaks, traffic, elem_steps=elems),
        "alg_bytes_per_step": alg,
        "gpu_launches": args.steps,
        "e2e": {"value": world * elems / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "clocks": clocks,
        "wall_s": round(wall, 3),
    }

    if rank == 0 and world == 1 and not args.headline_only:
        extras = {}
        for wspec in (I.MAMBA1P4B, I.LONGSEQ):
            t = time_scan(wspec, 10, 3, flush=True, cover=True)
            ms = statistics.median(t)
            extras[wspec.name] = {
                "elem_steps_per_s": wspec.elem_steps / (ms * 1e-3), "kernel_ms_median": ms,
                "roofline": roofline_obj(scan_alg_bytes(wspec), ms, peaks, profiled_traffic("scan_fwd_" + wspec.name),
                                         elem_steps=wspec.elem_steps)}
        t = time_scan(I.TINY, 20, 3, flush=False, cover=True)
        extras[I.TINY.name] = {"elem_steps_per_s": I.TINY.elem_steps / (statistics.median(t) * 1e-3),
                               "kernel_ms_median": statistics.median(t), "note": "launch-bound; parity case"}
        bms = time_bwd(HEADLINE, 10, 3)
        bro = roofline_obj(bwd_alg_bytes(HEADLINE), bms, peaks, profiled_traffic("scan_bwd_" + HEADLINE.name))
        mufu = peaks["sms"] * 32 / 3 * peaks["sm_max_mhz"] * 1e6
        bro["alu_ceiling"] = {"elem_steps_per_s": mufu, "achieved": HEADLINE.elem_steps / (bms * 1e-3),
                              "frac": round(HEADLINE.elem_steps / (bms * 1e-3) / mufu, 4),
                              "derivation": "three exponentials per element-step (forward walk, recompute, "
                                            "adjoint): %d SMs x 32/3 element-steps/clk x %.0f MHz"
                                            % (peaks["sms"], peaks["sm_max_mhz"])}
        extras["bwd_" + HEADLINE.name] = {
            "elem_steps_per_s": HEADLINE.elem_steps / (bms * 1e-3), "kernel_ms_median": bms,
            "roofline": bro, "note": "backward pass (all gradients, states recomputed), L2 flushed before each"}
        lbms = time_bwd(I.LONGSEQ, 3, 3)
        extras["bwd_" + I.LONGSEQ.name] = {
            "elem_steps_per_s": I.LONGSEQ.elem_steps / (lbms * 1e-3), "kernel_ms_median": lbms,
            "roofline": roofline_obj(bwd_alg_bytes(I.LONGSEQ), lbms, peaks, profiled_traffic("scan_bwd_" + I.LONGSEQ.name)),
            "note": "backward pass on the long sequence (batch 1, d_inner 2048, L 131072): 64 channel groups "
                    "walk the whole row each way, L2 flushed before each"}
        vbms = time_bwd(HEADLINE, 10, 3, variant=True)
        extras["bwd_reverse_starts_" + HEADLINE.name] = {
            "elem_steps_per_s": HEADLINE.elem_steps / (vbms * 1e-3), "kernel_ms_median": vbms,
            "roofline": roofline_obj(bwd_alg_bytes(HEADLINE) + HEADLINE.batch * HEADLINE.L, vbms, peaks,
                                     profiled_traffic("scan_bwd_reverse_starts_" + HEADLINE.name)),
            "note": "backward of the reverse-direction scan with a sequence start every 250 steps "
                    "(ss_scan_bwd_ex_*), L2 flushed before each"}
        tbms, tfms = time_bwd(HEADLINE, 10, 3, from_forward=True)
        extras["train_step_" + HEADLINE.name] = {
            "fwd_train_ms_median": tfms, "bwd_from_forward_ms_median": tbms,
            "elem_steps_per_s": HEADLINE.elem_steps / ((tfms + tbms) * 1e-3),
            "note": "training forward (also stores the state at every 16th step) + backward that starts from "
                    "those states; L2 flushed before each launch"}
        sspec = I.MAMBA2_LAYER
        sms2 = time_ssd(sspec, 10, 3)
        sby, sfl = ssd_alg(sspec)
        sro = roofline_obj(sby, sms2, peaks, profiled_traffic("ssd_chunk_" + sspec.name))
        tens = sfl / (sms2 * 1e-3) / 1e12
        sro["tensor"] = {"achieved_tflops": round(tens, 1), "peak_tflops": peaks["bf16_tflops"],
                         "frac": round(tens / peaks["bf16_tflops"], 4), "flops": sfl,
                         "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, burst)"}
        extras["ssd_" + sspec.name] = {
            "elem_steps_per_s": sspec.elem_steps / (sms2 * 1e-3), "kernel_ms_median": sms2, "roofline": sro,
            "note": "Mamba-2 scalar-decay scan: C B^T and the chunk walk on the tcgen05 tensor cores (TMEM "
                    "accumulators, 128-byte swizzled tensor-copy operands)"}
        cms, cbytes = time_conv(HEADLINE, 10, 3)
        extras["conv1d_silu_k4_" + HEADLINE.name] = {
            "elems_per_s": HEADLINE.batch * HEADLINE.d_inner * HEADLINE.L / (cms * 1e-3), "kernel_ms_median": cms,
            "roofline": roofline_obj(cbytes, cms, peaks, profiled_traffic("conv1d_silu_k4_" + HEADLINE.name)),
            "note": "causal depthwise conv (k = 4) + SiLU on the layer's (batch, d_inner, L) input, history out"}
        sms_, sbytes, scopy = time_conv_step(I.DECODE, 20)
        extras["conv_state_update_k4_" + I.DECODE.name] = {
            "ms_per_token": sms_,
            "roofline": roofline_obj(sbytes, sms_, peaks, profiled_traffic("conv_state_update_k4_" + I.DECODE.name)),
            "copy_floor": {"ms": scopy, "frac": sbytes / (scopy * 1e-3) / 1e9 / peaks["hbm_gbs"]},
            "note": "one decode step of the convolution (cache of 3 inputs per channel), L2 flushed before each; "
                    "copy_floor: a device copy of the same bytes (half read, half written) under the same protocol"}
        gms, fms = time_decode(I.DECODE, reps=3, warmup=3)
        dbytes = decode_alg_bytes(I.DECODE)
        extras[I.DECODE.name] = {
            "elem_steps_per_s": I.DECODE.elem_steps_per_step / (gms * 1e-3),
            "ms_per_token_graph": gms, "ms_per_token_l2_flushed": fms,
            "roofline_graph": roofline_obj(dbytes, gms, peaks, None),
            "roofline_l2_flushed": roofline_obj(dbytes, fms, peaks, profiled_traffic("state_update_" + I.DECODE.name)),
            "note": "graph: 1024 updates back to back, the 84 MB fp32 state can stay in the 126 MB L2; "
                    "l2_flushed: each update after the flush (256 MB written, then 256 MB read)"}
        line["workloads"] = extras

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, cores, desc, sec = oracle_rate(spec, budget_s=12.0)
        line["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
                                "seconds": round(sec, 2),
                                "single_thread_value": oracle_single_thread_rate(spec),
                                "single_thread_sample": "the first 16 (batch, channel) rows, one thread"}

    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
