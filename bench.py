#!/usr/bin/env python3
"""Benchmark of the B300 selective scan.

One step = one ssm_scan_fwd call over the 1M-token workload (batch 1,
d_inner 2048, d_state 16, L = 1,048,576; bf16 u/Δraw/z/B/C/out, fp32 state):
softplus, ZOH discretisation, recurrence, readout, D skip and SiLU gate, fused.
Prints one JSON line.  Also reported in the same line: the decode step
(ssm_step, batch 256 × d_inner 5120 × 16 states, 1000 steps), the end-to-end
throughput through the C ABI with inputs copied from pinned host memory and
the output read back, and the CPU oracle timed on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 run under torchrun (one process per GPU); each rank scans its own
workload-sized problem (independent rows, no collective): weak scaling.
``--impl reference`` times the CPU oracle (the slow plain definition) on the
host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "scan GB/s & channel·tokens/s (fraction of HBM roofline); ssm_step tokens/s"
WORKLOAD = "long_1m"
HBM_PEAK_FALLBACK = 6400.0
# FP32 lane operations of one state update (b, c, t, n) on the minimal path:
# Δ·A, Ā-1, x·(1/A), (x/A)·B + h, (Ā-1)·s + h, C·h accumulate (the exp is on the MUFU pipe).
FP32_OPS_PER_UPDATE = 6
SCAN_PROFILE = os.path.join(ROOT, "profiles", "scan_stream_kernel_long_seq.md")
SCAN_KERNEL_SRC = os.path.join(ROOT, "selective_state_space_154_b300", "csrc", "scan_stream.cu")


def source_digest(path):
    import hashlib
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def scan_traffic_per_launch():
    """DRAM bytes (read + write) per launch of the scan kernel on the 1M-token workload,
    from the committed ncu summary of the kernel, or None when the summary was taken
    on another version of the kernel source (its digest is recorded beside the figure)."""
    import re
    try:
        text = open(SCAN_PROFILE).read()
    except OSError:
        return None, "no committed capture"
    m = re.search(r"traffic_per_launch_bytes:\s*([0-9.eE+]+)", text)
    d = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    if not m or not d:
        return None, "capture summary lacks the figure or the source digest"
    if d.group(1) != source_digest(SCAN_KERNEL_SRC):
        return None, "kernel changed since the capture"
    return float(m.group(1)), f"ncu capture summarised in profiles/{os.path.basename(SCAN_PROFILE)}"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f)
    except OSError:
        return {}


def scan_alg_bytes(shape: W.ScanShape) -> int:
    """Bytes the scan must move: u, Δraw, z read and out written once per
    (batch, channel, token); B and C once per (batch, token); final state,
    A, D and bias once."""
    e = 2 if shape.dtype == torch.bfloat16 else 4
    ct = shape.batch * shape.d_inner * shape.seqlen
    return (4 * ct * e + 2 * shape.batch * shape.seqlen * shape.d_state * e
            + 4 * shape.batch * shape.d_inner * shape.d_state
            + 4 * shape.d_inner * shape.d_state + 8 * shape.d_inner)


def step_alg_bytes(shape: W.DecodeShape) -> int:
    e = 2 if shape.dtype == torch.bfloat16 else 4
    rows = shape.batch * shape.d_inner
    return (8 * rows * shape.d_state + 4 * rows * e + 2 * shape.batch * shape.d_state * e
            + 4 * shape.d_inner * shape.d_state + 8 * shape.d_inner)


# ---------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local
    return 0, 1, 0


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Each rank scans its own workload-sized problem drawn from its own seed."""
    return rank


def aggregate_throughput(units_per_rank_per_step: int, world: int, steps: int, max_secs: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank_per_step * steps / max_secs


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"ssm_bench_clocks_{os.getpid()}_{gpu_index}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    mhz.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "samples": len(mhz), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- timing helpers
class L2Flush:
    """Evict L2 between timed calls: write a 512 MiB buffer (4x the 126 MB L2),
    then read another one, so that the written lines are already back in HBM
    and the next timed call does not pay for their write-back."""

    def __init__(self, dev):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(128 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def time_steps(fn, steps, warmup, world, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / 1e3  # seconds


# ---------------------------------------------------------------- our arm
def bench_scan(args, rank, world, dev):
    import selective_state_space_154_b300 as ssm
    shape = W.SCAN_SHAPES[WORKLOAD]
    inp = W.scan_inputs(shape, device=dev, seed=rank_seed(rank))
    out = torch.empty_like(inp["u"])
    fs = torch.empty((shape.batch, shape.d_inner, shape.d_state), dtype=torch.float32, device=dev)
    ws_bytes = ssm.ssm_scan_workspace_bytes(shape.batch, shape.d_inner, shape.d_state, shape.seqlen, shape.dtype)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                         inp["bias"], out, fs, workspace=ws, stream=stream)

    with ClockSampler(torch.cuda.current_device()) as clk:
        secs = time_steps(step, args.steps, args.warmup, world, stream)
    status = ssm.ssm_scan_check(ws)
    if status != ssm.SSM_OK:
        raise RuntimeError(f"scan reported {ssm.ssm_status_string(status)}")
    return shape, inp, out, secs, clk.summary()


E2E_PIECE_TOKENS = 1 << 16


def bench_e2e(args, shape, inp, out, dev, world):
    """Same workload through the public API with the sequence in pinned host memory:
    ssm_scan_fwd_host copies u, delta, z, B, C in, scans and copies out back in pieces of
    E2E_PIECE_TOKENS tokens, the copies of one piece on their own streams overlapping
    the scan of another.  Wall clock per step, including every copy."""
    import selective_state_space_154_b300 as ssm
    names = ["u", "delta", "z", "B", "C"]
    host = {k: torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True) for k in names}
    for k in names:
        host[k].copy_(inp[k])
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    staging = torch.empty(ssm.ssm_scan_fwd_host_staging_bytes(shape.batch, shape.d_inner, shape.d_state,
                                                              shape.seqlen, E2E_PIECE_TOKENS, shape.dtype),
                          dtype=torch.uint8, device=dev)
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = out_host.numel() * out_host.element_size()
    stream = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    steps = max(1, min(args.steps, 5))

    def one():
        ssm.ssm_scan_fwd_host(host["u"], host["delta"], inp["A"], host["B"], host["C"], inp["D"], host["z"],
                              inp["bias"], out_host, piece_len=E2E_PIECE_TOKENS, staging=staging, stream=stream,
                              h2d_stream=s_in, d2h_stream=s_out)

    one()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
        stream.synchronize()
    secs = time.perf_counter() - t0
    secs = max_over_ranks(secs, world, dev)
    del host, out_host, staging
    return steps, secs, h2d, d2h


def bench_workloads(dev, runs=20):
    """The other scan workloads, one call each timed alone with L2 flushed before
    it (CUDA events around the call only); median of `runs`."""
    import selective_state_space_154_b300 as ssm
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    for name in ("tiny_fp32", "mamba130m_layer", "mamba2p8b_layer"):
        shape = W.SCAN_SHAPES[name]
        inp = W.scan_inputs(shape, device=dev, seed=0)
        out = torch.empty_like(inp["u"])
        fs = torch.empty((shape.batch, shape.d_inner, shape.d_state), dtype=torch.float32, device=dev)
        ws = torch.empty(max(16, ssm.ssm_scan_workspace_bytes(shape.batch, shape.d_inner, shape.d_state,
                                                              shape.seqlen, shape.dtype)), dtype=torch.uint8,
                         device=dev)

        def call():
            ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                             inp["bias"], out, fs, workspace=ws, stream=stream)

        for _ in range(3):
            call()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
        for a, b in evs:
            flush()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
        if ssm.ssm_scan_check(ws) != ssm.SSM_OK:
            raise RuntimeError(f"{name}: scan reported an error")
        secs = statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3
        alg = scan_alg_bytes(shape)
        res[name] = {"batch": shape.batch, "d_inner": shape.d_inner, "d_state": shape.d_state,
                     "seq_len": shape.seqlen, "io_dtype": "bf16" if shape.dtype == torch.bfloat16 else "fp32",
                     "us": secs * 1e6, "channel_tokens_per_s": shape.channel_tokens / secs,
                     "gbs": alg / secs / 1e9, "alg_bytes": alg}
        del inp, out, fs, ws
    return res


def bench_scan_bwd(dev, hbm_peak, runs=10):
    """Backward of the scan on the two training-shaped layers, each call timed
    alone after an L2 flush (median).  Algorithmic bytes: u, delta, z, dout read and
    du, delta and z gradients written once per (batch, channel, token), B and C read
    and their fp32 gradients written once per (batch, token, state)."""
    import selective_state_space_154_b300 as ssm
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    res = {"note": "states recomputed from checkpoints every 8 tokens (workspace); the sequence is split "
                   "into chunks combined from per-chunk summaries (two launches); median of 10, L2 flushed "
                   "before each; deterministic_us: ssm_scan_bwd_deterministic (partial sums reduced in a fixed "
                   "order by a third launch)"}
    for name in ("mamba130m_layer", "mamba2p8b_layer"):
        shape = W.SCAN_SHAPES[name]
        inp = W.scan_inputs(shape, device=dev, seed=0)
        gen = torch.Generator(device=dev).manual_seed(1)
        dout = torch.randn(inp["u"].shape, generator=gen, device=dev).to(shape.dtype)
        g = dict(du=torch.empty_like(inp["u"]), ddelta=torch.empty_like(inp["u"]), dz=torch.empty_like(inp["u"]),
                 dA=torch.empty_like(inp["A"]), dB=torch.empty(inp["B"].shape, device=dev),
                 dC=torch.empty(inp["C"].shape, device=dev), dD=torch.empty_like(inp["D"]),
                 dbias=torch.empty(shape.d_inner, device=dev))
        ws = torch.empty(max(16, ssm.ssm_scan_bwd_deterministic_workspace_bytes(
            shape.batch, shape.d_inner, shape.d_state, shape.seqlen, shape.dtype)), dtype=torch.uint8, device=dev)

        def timed(det):
            def call():
                ssm.ssm_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                 inp["bias"], dout, g["du"], g["ddelta"], g["dA"], g["dB"], g["dC"], g["dD"], g["dz"],
                                 g["dbias"], workspace=ws, stream=stream, deterministic=det)

            call()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
            for a, b in evs:
                flush()
                a.record(stream)
                call()
                b.record(stream)
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3

        secs = timed(False)
        secs_det = timed(True)
        ct = shape.channel_tokens
        alg = 7 * ct * 2 + shape.batch * shape.seqlen * shape.d_state * (2 * 2 + 2 * 4)
        res[name] = {"batch": shape.batch, "d_inner": shape.d_inner, "d_state": shape.d_state,
                     "seq_len": shape.seqlen, "us": secs * 1e6, "channel_tokens_per_s": ct / secs,
                     "gbs": alg / secs / 1e9, "hbm_frac": alg / secs / 1e9 / hbm_peak, "alg_bytes": alg,
                     "deterministic_us": secs_det * 1e6}
        del inp, dout, g, ws
    return res


def conv_alg_bytes(rows, L, width, esz):
    """x read and out written once per (row, token), the carried state read and
    the final state written once per row (weight and bias are added by the caller)."""
    return rows * L * 2 * esz + 2 * rows * (width - 1) * esz



def ssd_alg(shape):
    """Algorithmic bytes and tensor FLOPs of one Mamba-2 layer scan: x and z read and
    out written once per (batch, token, head, p), dt once per (batch, token, head), B
    and C once per (batch, token, group, n) (bf16); FLOPs of the chunked evaluation
    per (batch, head, 128-token chunk): S = C Bᵀ (2·Q·Q·N), Y = G X and Y_in = C h_inᵀ
    (2·Q·P·Q + 2·Q·P·N) and the chunk state Bᵀ diag(w) X (2·N·P·Q), counting each
    operand once (the second bf16 term of G and of w·x is precision, not work)."""
    b, L, H, P, G, N = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.ngroups, shape.d_state
    q = 128
    nch = (L + q - 1) // q
    alg = 3 * 2 * b * L * H * P + 2 * b * L * H + 2 * 2 * b * L * G * N
    flops = b * H * nch * (2 * q * q * N + 2 * q * P * q + 2 * q * P * N + 2 * N * P * q)
    return alg, flops


def bench_ssd(dev, hbm_peak, tc_peak, runs=20):
    """The Mamba-2 (SSD) layer scan on the two Mamba-2-shaped layers, each call
    timed alone after an L2 flush (median)."""
    import selective_state_space_154_b300 as ssm
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    res = {"note": "chunks of 128 tokens on the tensor cores (tcgen05, bf16 operands, fp32 accumulators in "
                   "tensor memory); one launch, one CTA walking the sequence of each (batch, head) with the "
                   "state in registers; median of 20, L2 flushed before each; hbm_frac of the "
                   "measured copy bandwidth, tensor_frac of the measured cuBLAS bf16 burst"}
    for name in ("mamba2_130m_layer", "mamba2_2p7b_layer"):
        shape = W.SSD_SHAPES[name]
        inp = W.ssd_inputs(shape, device=dev, seed=0)
        out = torch.empty_like(inp["x"])
        fs = torch.empty((shape.batch, shape.nheads, shape.headdim, shape.d_state), device=dev)
        ws = torch.empty(ssm.ssd_scan_workspace_bytes(shape.batch, shape.seqlen, shape.nheads, shape.headdim,
                                                      shape.ngroups, shape.d_state), dtype=torch.uint8, device=dev)
        call = lambda: ssm.ssd_scan_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                        inp["dt_bias"], None, out, fs, workspace=ws, stream=stream)
        for _ in range(3):
            call()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
        for a, b in evs:
            flush()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
        secs = statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3
        if ssm.ssm_scan_check(ws) != 0:
            raise RuntimeError("ssd_scan_fwd reported a device-side timeout")
        alg, flops = ssd_alg(shape)
        res[name] = {"batch": shape.batch, "seq_len": shape.seqlen, "nheads": shape.nheads,
                     "headdim": shape.headdim, "ngroups": shape.ngroups, "d_state": shape.d_state,
                     "us": secs * 1e6, "channel_tokens_per_s": shape.channel_tokens / secs,
                     "gbs": alg / secs / 1e9, "hbm_frac": alg / secs / 1e9 / hbm_peak, "alg_bytes": alg,
                     "tflops": flops / secs / 1e12, "tensor_frac": flops / secs / 1e12 / tc_peak,
                     "workspace_bytes": ws.numel()}
        del inp, out, fs, ws
    # decode: one token for 256 sequences of the 2.7B-shaped layer (80 heads × 64 × 128 fp32 state,
    # 671 MB > L2, so no flush is needed), steps timed one by one
    b, H, P, N = 256, 80, 64, 128
    dshape = W.SsdShape("decode", b, 1, H, P, 1, N, torch.bfloat16)
    dinp = W.ssd_inputs(dshape, device=dev, seed=0)
    state = torch.zeros((b, H, P, N), device=dev)
    tok = dict(x=dinp["x"][:, 0].contiguous(), dt=dinp["dt"][:, 0].contiguous(), B=dinp["B"][:, 0].contiguous(),
               C=dinp["C"][:, 0].contiguous(), z=dinp["z"][:, 0].contiguous())
    yout = torch.empty_like(tok["x"])
    step = lambda: ssm.ssd_step(state, tok["x"], tok["dt"], dinp["A"], tok["B"], tok["C"], D=dinp["D"], z=tok["z"],
                                dt_bias=dinp["dt_bias"], out=yout, stream=stream)
    for _ in range(3):
        step()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
    for a, e in evs:
        a.record(stream)
        step()
        e.record(stream)
    torch.cuda.synchronize()
    secs = statistics.median(a.elapsed_time(e) for a, e in evs) / 1e3
    alg = 2 * b * H * P * N * 4 + 3 * b * H * P * 2 + b * H * 2 + 2 * b * N * 2
    res["decode_mamba2_2p7b"] = {"batch": b, "nheads": H, "headdim": P, "d_state": N, "us": secs * 1e6,
                                 "tokens_per_s": b / secs, "gbs": alg / secs / 1e9,
                                 "hbm_frac": alg / secs / 1e9 / hbm_peak, "alg_bytes": alg,
                                 "note": "ssd_step, state read and written in place (671 MB > L2)"}
    return res


def bench_conv(dev, hbm_peak, runs=20):
    """Causal Conv1D + SiLU: the sequence form on the 2.8B-shaped layer's x (L2
    flushed before each call) and on the 1M-token rows (larger than L2), and the
    decode step on the decode workload's rows (L2 flushed before each step)."""
    import selective_state_space_154_b300 as ssm
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    res = {"width": W.CONV_WIDTH,
           "note": "each call timed alone with CUDA events, median; hbm_frac of the measured copy bandwidth"}

    def timed(call, n, flush_each=True):
        for _ in range(3):
            call()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            if flush_each:
                flush()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3

    for name in ("mamba2p8b_layer", "long_1m"):
        shape = W.SCAN_SHAPES[name]
        cv = W.conv_inputs(shape.batch, shape.d_inner, shape.seqlen, device=dev, seed=0)
        out = torch.empty_like(cv["x"])
        fs = torch.empty_like(cv["state"])
        call = lambda: ssm.ssm_conv1d_fwd(cv["x"], cv["w"], cv["bias"], cv["state"], out, fs, stream=stream)
        secs = timed(call, runs if name != "long_1m" else 5, flush_each=name != "long_1m")
        alg = conv_alg_bytes(shape.rows, shape.seqlen, W.CONV_WIDTH, 2) + shape.d_inner * (W.CONV_WIDTH + 1) * 4
        res[f"fwd_{name}"] = {"batch": shape.batch, "d_inner": shape.d_inner, "seq_len": shape.seqlen,
                              "us": secs * 1e6, "channel_tokens_per_s": shape.channel_tokens / secs,
                              "gbs": alg / secs / 1e9, "hbm_frac": alg / secs / 1e9 / hbm_peak, "alg_bytes": alg}
        del cv, out, fs
    shape = W.DECODE_SHAPE
    cv = W.conv_inputs(shape.batch, shape.d_inner, 1, device=dev, seed=0)
    x = cv["x"][:, :, 0].contiguous()
    out = torch.empty_like(x)
    st = cv["state"]
    secs = timed(lambda: ssm.ssm_conv1d_step(st, x, cv["w"], cv["bias"], out, stream=stream), 200)
    rows = shape.batch * shape.d_inner
    alg = 2 * rows * 2 + 2 * rows * (W.CONV_WIDTH - 1) * 2 + shape.d_inner * (W.CONV_WIDTH + 1) * 4
    res["step_decode"] = {"batch": shape.batch, "d_inner": shape.d_inner, "us": secs * 1e6,
                          "tokens_per_s": shape.batch / secs, "gbs": alg / secs / 1e9,
                          "hbm_frac": alg / secs / 1e9 / hbm_peak, "alg_bytes": alg}
    return res


def bench_decode(dev):
    """ssm_step on the decode workload: each timed step starts with L2 flushed
    (in a model, the other layers evict this layer's state between its steps);
    also the same 1000 steps back to back in one CUDA graph (state warm in L2)."""
    import selective_state_space_154_b300 as ssm
    shape = W.DECODE_SHAPE
    inp = W.decode_inputs(shape, device=dev, seed=0)
    state = torch.zeros((shape.batch, shape.d_inner, shape.d_state), dtype=torch.float32, device=dev)
    out = torch.empty((shape.batch, shape.d_inner), dtype=shape.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)

    def step(s):
        ssm.ssm_step(state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s], inp["C"][s], inp["D"],
                     inp["z"][s], inp["bias"], out, stream=stream)

    for s in range(5):
        step(s)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(shape.steps)]
    for s in range(shape.steps):
        flush()
        evs[s][0].record(stream)
        step(s)
        evs[s][1].record(stream)
    torch.cuda.synchronize()
    cold = sum(a.elapsed_time(b) for a, b in evs) / 1e3
    # warm: the whole 1000-step decode captured once as a graph
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step(0)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            for s in range(shape.steps):
                ssm.ssm_step(state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s], inp["C"][s], inp["D"],
                             inp["z"][s], inp["bias"], out, stream=side)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    warm = e0.elapsed_time(e1) / 1e3
    per_step_bytes = step_alg_bytes(shape)
    return {
        "metric": "ssm_step tokens/s", "unit": "tokens/s",
        "value": shape.batch * shape.steps / cold,
        "us_per_step": cold / shape.steps * 1e6,
        "gbs": per_step_bytes * shape.steps / cold / 1e9,
        "alg_bytes_per_step": per_step_bytes,
        "l2": "flushed (512 MiB write, then 512 MiB read) before every timed step; steps timed one by one with CUDA events",
        "warm_l2_graph": {"value": shape.batch * shape.steps / warm, "us_per_step": warm / shape.steps * 1e6,
                          "gbs": per_step_bytes * shape.steps / warm / 1e9,
                          "note": "1000 steps replayed back to back as one CUDA graph; the 84 MB state stays in L2"},
        "config": {"workload": "decode", "batch": shape.batch, "d_inner": shape.d_inner,
                   "d_state": shape.d_state, "steps": shape.steps, "io": "bf16", "state": "fp32"},
        "gpu_launches": shape.steps,
    }


# ---------------------------------------------------------------- CPU oracle
def cpu_threads():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def make_oracle_rows(shape, rows, length, seed=0):
    """Host float64 inputs of `rows` channels × `length` tokens of the workload
    (drawn on the GPU when available, else on the CPU, then rounded as the GPU sees them)."""
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    sub = W.ScanShape("sample", 1, rows, shape.d_state, length, shape.dtype)
    inp = W.scan_inputs(sub, device=dev, seed=seed)
    f = lambda t: None if t is None else t.detach().to("cpu", torch.float64).numpy()
    return [f(inp["u"]), f(inp["delta"]), f(inp["A"]), f(inp["B"]), f(inp["C"]), f(inp["D"]), f(inp["z"]),
            f(inp["bias"])]


def _oracle_call(args_list, threads):
    import oracle
    u, delta, A, B, C, D, z, bias = args_list
    t0 = time.perf_counter()
    oracle.scan(u, delta, A, B, C, D=D, z=z, bias=bias, threads=threads)
    return time.perf_counter() - t0


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(target_s=12.0, rows=128):
    """The oracle as it stands on the host cores: a seeded subset of `rows` channels of
    the workload at full length, threaded over channels on every core, repeated until
    about target_s of work has been timed; and one full-length channel on one core."""
    shape = W.SCAN_SHAPES[WORKLOAD]
    threads = cpu_threads()
    length = shape.seqlen
    sample = make_oracle_rows(shape, rows, length, seed=1)
    total, calls = 0.0, 0
    while total < target_s and calls < 100:
        total += _oracle_call(sample, threads)
        calls += 1
    u, delta, A, B, C, D, z, bias = sample
    cut = lambda a, sl: None if a is None else a[sl]
    one = [u[:, :1], delta[:, :1], A[:1], B, C, cut(D, slice(0, 1)), cut(z, (slice(None), slice(0, 1))),
           cut(bias, slice(0, 1))]
    single = _oracle_call(one, 1)
    return {"value": rows * length * calls / total, "unit": "channel·tokens/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(), "seconds": total,
            "single_core": {"value": length / single, "unit": "channel·tokens/s",
                            "sample": f"1 channel x {length} tokens on 1 thread"},
            "sample": f"seeded subset of {rows} channels x {length} tokens (full length) of the {WORKLOAD} workload "
                      f"(d_state {shape.d_state}, bf16-rounded inputs, float64 arithmetic), oracle.scan threaded "
                      f"over channels on {threads} threads, run {calls} times"}


# ---------------------------------------------------------------- arms
def run_ours(args):
    rank, world, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the reference arm runs on CPU: --impl reference)")
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = measured_peaks()
    shape, inp, out, secs, clocks = bench_scan(args, rank, world, dev)
    secs = max_over_ranks(secs, world, dev)
    ct = shape.channel_tokens
    value = aggregate_throughput(ct, world, args.steps, secs)
    ms = secs / args.steps * 1e3
    alg = scan_alg_bytes(shape)
    gbs = alg / (secs / args.steps) / 1e9
    sm_mhz = clocks.get("sm_mhz") or peaks.get("sm_max_mhz", 2032.0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rates = probe_pipe_rates(threads_list=(512,)) if rank == 0 else None
    fp32_lanes = rates["ffma2 (packed f32x2)"]["512"] if rates else 128.0
    alu_peak = sms * fp32_lanes * sm_mhz * 1e6 / 1e12
    alu_achieved = FP32_OPS_PER_UPDATE * ct * shape.d_state / (secs / args.steps) / 1e12
    traffic, traffic_note = scan_traffic_per_launch()
    hbm_peak = peaks.get("hbm_gbs")
    hbm_note = "of measured" if hbm_peak else "of fallback"
    hbm_peak = hbm_peak or HBM_PEAK_FALLBACK

    e2e_steps, e2e_secs, h2d, d2h = bench_e2e(args, shape, inp, out, dev, world)
    del inp, out
    torch.cuda.empty_cache()
    decode = bench_decode(dev) if rank == 0 else None
    others = bench_workloads(dev) if rank == 0 else None
    conv = bench_conv(dev, hbm_peak) if rank == 0 else None
    bwd = bench_scan_bwd(dev, hbm_peak) if rank == 0 else None
    ssd = bench_ssd(dev, hbm_peak, peaks.get("bf16_tflops")) if rank == 0 else None
    cpu = cpu_baseline() if (rank == 0 and world == 1) else None

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "channel·tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{WORKLOAD} scan: batch {shape.batch}, d_inner {shape.d_inner}, "
                                   f"d_state {shape.d_state}, L {shape.seqlen}; bf16 u/delta/z/B/C/out, "
                                   "fp32 A/D/bias/state, softplus+ZOH+recurrence+readout+D+silu gate fused",
                       "batch": shape.batch, "d_inner": shape.d_inner, "d_state": shape.d_state,
                       "seq_len": shape.seqlen, "io_dtype": "bf16",
                       "parallelism": "one independent problem per GPU, no collective" if world > 1 else "single GPU",
                       "l2": "inputs 17.2 GB > 126 MB L2 (no flush needed)"},
            "gbs": gbs,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "traffic": traffic, "peak_note": hbm_note + " (MEASURED_PEAKS.json hbm_gbs, burst copy)",
                         "achieved_basis": f"algorithmic bytes {alg} per launch (u, delta, z read and out written once "
                                           "per channel-token; B, C once per token; final state, A, D, bias once) / "
                                           "CUDA-event time per launch",
                         "traffic_note": traffic_note,
                         "alu": {"achieved": alu_achieved, "peak": alu_peak, "unit": "FP32 Tops/s",
                                 "frac": alu_achieved / alu_peak,
                                 "achieved_basis": f"{FP32_OPS_PER_UPDATE} FP32 lane operations per state update x "
                                                   f"{ct * shape.d_state} updates per launch",
                                 "peak_basis": f"{sms} SMs x {fp32_lanes:.1f} FP32 lane-ops per SM-clock (measured "
                                               f"now by the pipe-rate probe, packed FFMA2) x {sm_mhz:.0f} MHz (median SM "
                                               "clock sampled during the timed region)",
                                 "pipe_rates": rates}},
            "e2e": {"value": world * ct * e2e_steps / e2e_secs, "unit": "channel·tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "note": "public API ssm_scan_fwd_host: the sequence in pinned host memory, copied in, scanned and "
                            f"copied out in pieces of {E2E_PIECE_TOKENS} tokens, copies overlapped with the scans on "
                            "separate streams; wall clock per step, every copy inside"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "decode": decode,
            "workloads": {"note": "other scan workloads, each call timed alone after an L2 flush (512 MiB write, then 512 MiB read), "
                                  "median of 20; hbm_frac of the measured copy bandwidth",
                          **({k: dict(v, hbm_frac=v["gbs"] / hbm_peak) for k, v in others.items()}
                             if others else {})},
            "conv1d": conv,
            "scan_bwd": bwd,
            "ssd": ssd,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile_case(args):
    """A short run of one kernel for ncu captures (prints timing, not the JSON line)."""
    import selective_state_space_154_b300 as ssm
    dev = torch.device("cuda", 0)
    if args.only == "scan":
        base = W.SCAN_SHAPES[args.workload]
        shape = W.ScanShape(base.name, args.batch or base.batch, args.dinner or base.d_inner, base.d_state,
                            args.seqlen or base.seqlen, base.dtype)
        inp = W.scan_inputs(shape, device=dev, seed=0)
        out = torch.empty_like(inp["u"])
        ws = torch.empty(max(16, ssm.ssm_scan_workspace_bytes(shape.batch, shape.d_inner, shape.d_state,
                                                              shape.seqlen, shape.dtype)), dtype=torch.uint8, device=dev)
        fn = lambda: ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                      inp["bias"], out, None, workspace=ws)
        units = shape.channel_tokens
    elif args.only == "bwd":
        base = W.SCAN_SHAPES[args.workload]
        shape = W.ScanShape(base.name, base.batch, args.dinner or base.d_inner, base.d_state, args.seqlen or base.seqlen,
                            base.dtype)
        inp = W.scan_inputs(shape, device=dev, seed=0)
        gen = torch.Generator(device=dev).manual_seed(1)
        dout = torch.randn(inp["u"].shape, generator=gen, device=dev).to(shape.dtype)
        gr = dict(du=torch.empty_like(inp["u"]), ddelta=torch.empty_like(inp["u"]), dz=torch.empty_like(inp["u"]),
                  dA=torch.empty_like(inp["A"]), dB=torch.empty(inp["B"].shape, device=dev),
                  dC=torch.empty(inp["C"].shape, device=dev), dD=torch.empty_like(inp["D"]),
                  dbias=torch.empty(shape.d_inner, device=dev))
        ws = torch.empty(max(16, ssm.ssm_scan_bwd_workspace_bytes(shape.batch, shape.d_inner, shape.d_state,
                                                                  shape.seqlen, shape.dtype)), dtype=torch.uint8,
                         device=dev)
        fn = lambda: ssm.ssm_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                      inp["bias"], dout, gr["du"], gr["ddelta"], gr["dA"], gr["dB"], gr["dC"],
                                      gr["dD"], gr["dz"], gr["dbias"], workspace=ws)
        units = shape.channel_tokens
    elif args.only == "ssd":
        shape = W.SSD_SHAPES[args.workload if args.workload in W.SSD_SHAPES else "mamba2_2p7b_layer"]
        if args.seqlen:
            shape = W.SsdShape(shape.name, shape.batch, args.seqlen, shape.nheads, shape.headdim, shape.ngroups,
                               shape.d_state, shape.dtype)
        inp = W.ssd_inputs(shape, device=dev, seed=0)
        out = torch.empty_like(inp["x"])
        ws = torch.empty(ssm.ssd_scan_workspace_bytes(shape.batch, shape.seqlen, shape.nheads, shape.headdim,
                                                      shape.ngroups, shape.d_state), dtype=torch.uint8, device=dev)
        fn = lambda: ssm.ssd_scan_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                      inp["dt_bias"], None, out, None, workspace=ws)
        units = shape.channel_tokens
    elif args.only == "conv":
        base = W.SCAN_SHAPES[args.workload]
        L = args.seqlen or base.seqlen
        cv = W.conv_inputs(base.batch, args.dinner or base.d_inner, L, device=dev, seed=0)
        out = torch.empty_like(cv["x"])
        fs = torch.empty_like(cv["state"])
        fn = lambda: ssm.ssm_conv1d_fwd(cv["x"], cv["w"], cv["bias"], cv["state"], out, fs)
        units = cv["x"].numel()
    else:
        shape = W.DECODE_SHAPE
        inp = W.decode_inputs(shape, device=dev, seed=0, steps=8)
        state = torch.zeros((shape.batch, shape.d_inner, shape.d_state), device=dev)
        out = torch.empty((shape.batch, shape.d_inner), dtype=shape.dtype, device=dev)
        fn = lambda: ssm.ssm_step(state, inp["x"][0], inp["delta"][0], inp["A"], inp["B"][0], inp["C"][0],
                                  inp["D"], inp["z"][0], inp["bias"], out)
        units = shape.batch
    secs = time_steps(fn, args.steps, args.warmup, 1, torch.cuda.current_stream(dev))
    print(f"{args.only}: {secs / args.steps * 1e3:.4f} ms per call, {units * args.steps / secs:.4e} units/s")


PROBE_VARIANTS = {0: ("ffma", "FP32 lane-ops"), 1: ("ffma2 (packed f32x2)", "FP32 lane-ops"),
                  2: ("mufu ex2", "ex2"), 3: ("scan state update, packed", "state updates"),
                  4: ("scan state update, scalar", "state updates"), 5: ("alu prmt+lop3", "ALU lane-ops"),
                  6: ("12 ffma2 + 4 ex2 chains", "rounds (12 ffma2 + 4 ex2 each)"),
                  7: ("6 ffma2 + 4 ex2 chains", "rounds (6 ffma2 + 4 ex2 each)"),
                  8: ("scan state update, packed, ex2 replaced by fmul", "state updates"),
                  9: ("scan token, 1 thread/row, 8 tokens unrolled", "state updates"),
                  10: ("scan token, 1 thread/row, 4 tokens unrolled", "state updates"),
                  11: ("scan token, 2 threads/row, 8 tokens unrolled", "state updates"),
                  12: ("scan token, 1 thread/row, ex2 one token ahead", "state updates"),
                  13: ("scan token, 1 thread/row, ex2 one token ahead, unrolled x2", "state updates")}


PROBE_THREADS = {3: (512, 640), 4: (512,), 8: (512,), 9: (512, 640), 10: (512, 640), 11: (512, 768, 1024),
                 12: (512, 640), 13: (512,)}


def probe_pipe_rates(threads_list=(512, 1024)):
    """Per-SM throughput of the arithmetic pipes, from the probe library: one CTA per
    SM, register-resident independent chains, each CTA timed by the SM clock counter.
    Returns {variant: {threads: work per SM-clock (median over CTAs)}}."""
    import ctypes
    from selective_state_space_154_b300 import build as ssm_build
    lib = ctypes.CDLL(ssm_build.build_probe())
    fn = lib.ssm_probe_pipe_rates
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_double)]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    res = {}
    for v, (name, unit) in PROBE_VARIANTS.items():
        res[name] = {"unit": f"{unit} per SM per clock"}
        for threads in (PROBE_THREADS.get(v, threads_list) if len(threads_list) > 1 else threads_list):
            iters = 2000 if v not in PROBE_THREADS else 400
            cyc = (ctypes.c_longlong * sms)()
            work = ctypes.c_double()
            for _ in range(2):  # the first run warms up
                rc = fn(v, sms, threads, iters, cyc, ctypes.byref(work))
                if rc != 0:
                    raise RuntimeError(f"probe {name}: CUDA error {rc}")
            per_sm = sorted(work.value * threads / c for c in cyc)
            res[name][str(threads)] = per_sm[len(per_sm) // 2]
    return res


def run_peaks(args):
    res = probe_pipe_rates()
    print(json.dumps({"pipe_rates": res}, indent=1), flush=True)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shape = W.SCAN_SHAPES[WORKLOAD]
    threads = cpu_threads()
    length = 1 << 17
    rows = threads * 4
    sample = make_oracle_rows(shape, rows, length, seed=0)
    for _ in range(args.warmup):
        _oracle_call(sample, threads)
    total = 0.0
    for _ in range(args.steps):
        total += _oracle_call(sample, threads)
    value = rows * length * args.steps / total
    desc = (f"each step: {rows} channels x {length} tokens of the {WORKLOAD} workload "
            f"(d_state {shape.d_state}), oracle.scan in float64 on {threads} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "channel·tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} scan (bounded sample, see cpu_baseline)", "batch": shape.batch,
                   "d_inner": shape.d_inner, "d_state": shape.d_state, "seq_len": shape.seqlen},
        "cpu_baseline": {"value": value, "unit": "channel·tokens/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "channel·tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", choices=["all", "scan", "decode", "conv", "bwd", "ssd", "peaks"], default="all",
                    help="profiling aid: run only the scan, the decode step, the Conv1D or the backward (no JSON line)")
    ap.add_argument("--seqlen", type=int, default=None,
                    help="profiling aid: scan another sequence length of the same workload")
    ap.add_argument("--batch", type=int, default=None,
                    help="profiling aid: scan another batch size of the same workload")
    ap.add_argument("--dinner", type=int, default=None,
                    help="profiling aid: scan another number of channels of the same workload")
    ap.add_argument("--workload", choices=sorted(W.SCAN_SHAPES) + sorted(W.SSD_SHAPES), default=WORKLOAD,
                    help="profiling aid: the workload --only scan / conv / bwd / ssd runs")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    elif args.only == "peaks":
        run_peaks(args)
    elif args.only != "all":
        run_profile_case(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
