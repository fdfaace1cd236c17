#!/usr/bin/env python3
"""Benchmark: shifted-window attention forward + backward on one GB300.

A step is one pass of the whole path over one batch of the depth3d workload
(16 levels x 192 x 384 tokens, C=256, 8 heads x 32, window 2x8x8, shift
(1,4,4), lon periodic, land mask growing with depth; bf16): swin_attn_fwd then
swin_attn_bwd (dQ, dK, dV, dBias). Every input tensor (604 MB each) is larger
than the 129 MB L2, so no flush runs between steps.

The same line carries `configs`: all five workloads (tiny_fp32, grid1deg,
ragged, eddy_ocean, depth3d) timed one launch at a time with a 1 GiB L2
flush before every launch, the median of >= 50 repetitions after >= 10
warm-ups, with each one's roofline fraction against its algorithmic bytes.

Prints one JSON line (rank 0). --impl reference times the CPU oracle on the
same workload instead (bounded samples of windows, fp64).
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

METRIC = "window-attention Mtokens/s fwd & fwd+bwd (bf16) and % of roofline, 1 GB300"
WORKLOAD = "depth3d"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def workload_counts(wl, win_src, land, lse_written=True):
    """Algorithmic FLOPs and bytes per launch, as the measurement section of
    the survey counts them: forward = 4 * B * sum over windows of (real
    slots)^2 * C FLOPs, backward = 2.5x that; forward bytes = Q, K, V in and O
    out (4 N C e) + LSE (4 N heads, when written) + land + bias; backward
    bytes = Q, K, V, O, dO in and dQ, dK, dV out (8 N C e) + LSE and delta
    (2 x 4 N heads) + land + bias in + dBias out. Returns (fwd_flop,
    bwd_flop, fwd_bytes, bwd_bytes, bwd_bytes_moved), where bwd_bytes_moved
    is what this backward actually has to move: it recomputes delta from P
    and dP, so it reads neither O nor delta (7 N C e + LSE + land + 2 bias)."""
    n_real = (win_src >= 0).sum(1).astype(np.float64)  # real slots per window
    N = wl.batch * wl.tokens
    C, H, e = wl.channels, wl.heads, 2 if wl.dtype == "bf16" else 4
    rows = int(np.prod([2 * w - 1 for w in wl.window]))
    fwd_flop = 4.0 * wl.batch * float((n_real ** 2).sum()) * C
    bwd_flop = 2.5 * fwd_flop
    land_b = N if land is not None else 0
    bias_b = rows * H * 4 if wl.bias else 0
    lse_b = 4 * N * H
    fwd_bytes = 4 * N * C * e + (lse_b if lse_written else 0) + land_b + bias_b
    bwd_bytes = 8 * N * C * e + 2 * lse_b + land_b + 2 * bias_b
    bwd_moved = 7 * N * C * e + lse_b + land_b + 2 * bias_b
    return fwd_flop, bwd_flop, fwd_bytes, bwd_bytes, bwd_moved


def roof_us(flop, nbytes, peaks):
    """Roofline time of one launch: the slower of the bf16 tensor-core time
    (burst peak) and the HBM time, both from the measured peaks."""
    return max(flop / (peaks["bf16_tflops"] * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9)) * 1e6


# per-config bars: forward >= 50 % and backward >= 35 % of the roofline (bf16)
TARGETS = {"tiny_fp32": None, "grid1deg": {"fwd": 0.50}, "ragged": {"fwd": 0.50, "bwd": 0.35},
           "eddy_ocean": {"fwd": 0.50, "bwd": 0.35}, "depth3d": {"fwd": 0.50, "bwd": 0.35}}
# timed beside the five configurations (no bar of its own): the large-window regime
EXTRA = ["terra_w32", "beast_w64k"]
# launches of one of these take a large part of a second: fewer repetitions
EXTRA_REPS = {"beast_w64k": (5, 2)}
NOTES = {"terra_w32": "windows of 1 024 tokens, head_dim 128: key-tiled tcgen05 kernels; tensor-bound",
         "beast_w64k": "windows of 64 800 tokens (507 key tiles), head_dim 128, no bias: key-tiled tcgen05 kernels; "
                       "tensor-bound; FLOPs count every pair of real slots of a window (regions included)",
         "tiny_fp32": "fp32 SIMT path, 512 tokens: launch-bound, parity only",
         "grid1deg": "forward only (inference: no LSE written, its bytes not counted)",
         "eddy_ocean": "not ragged: 256 = 32 x 8 rows divide into 8-row windows; irregular through the land mask"}
FLUSH_BYTES = 1 << 30
# largest window the CPU-baseline and parity legs run through the per-window oracle
ORACLE_WINDOW_SLOTS = 2048


def time_config(wl, x, peaks, flush, reps=50, warmup=10, kernels="auto"):
    """One workload timed launch by launch: before every launch a 1 GiB buffer
    is written (L2 flush), then CUDA events on the launching stream bracket
    the launch alone. Median over `reps` after `warmup` repetitions."""
    import torch
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    dev = torch.device("cuda", torch.cuda.current_device())
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch,
                               wl.dtype, wl.has_land, kernels)
    win_src = C.swin_attn_plan_tables(attn.plan)[0]
    fwd_flop, bwd_flop, fwd_bytes, bwd_bytes, bwd_moved = workload_counts(wl, win_src, x["land"],
                                                                         lse_written=wl.backward)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    d = {k_: torch.from_numpy(x[k_]).to(dev).to(tdt) for k_ in ("q", "k", "v", "dout")}
    bias = torch.from_numpy(x["bias"]).to(dev) if wl.bias else None
    land = torch.from_numpy(x["land"]).to(dev) if x["land"] is not None else None
    o = torch.empty(attn.shape, dtype=tdt, device=dev)
    lse = torch.empty(attn.lse_shape, dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty(attn.shape, dtype=tdt, device=dev) for _ in range(3))
    dbias = attn.new_bias() if wl.bias else None
    ws = attn.workspace()
    stream = torch.cuda.current_stream()
    fwd_t, bwd_t, bwdo_t = [], [], []
    backward = wl.backward
    # head_dim 128: the backward also given the forward's output (delta = dO . O)
    with_o = backward and wl.head_dim == 128
    if backward:
        try:  # a kernel family without a backward yet is timed forward only
            C.swin_attn_fwd(attn.plan, d["q"], d["k"], d["v"], bias, land, o, lse, stream)
            C.swin_attn_bwd(attn.plan, d["q"], d["k"], d["v"], d["dout"], lse, bias, land, dq, dk, dv, dbias, ws,
                            stream)
        except C.SwinAttnError as e:
            if e.code != C.SWIN_ERR_UNSUPPORTED:
                raise
            backward = False
    for r in range(warmup + reps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        flush.add_(1)
        ev[0].record(stream)
        C.swin_attn_fwd(attn.plan, d["q"], d["k"], d["v"], bias, land, o, lse if wl.backward else None, stream)
        ev[1].record(stream)
        if backward:
            flush.add_(1)
            ev[2].record(stream)
            C.swin_attn_bwd(attn.plan, d["q"], d["k"], d["v"], d["dout"], lse, bias, land, dq, dk, dv, dbias, ws,
                            stream)
            ev[3].record(stream)
        if with_o:
            ev += [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            flush.add_(1)
            ev[4].record(stream)
            C.swin_attn_bwd_o(attn.plan, d["q"], d["k"], d["v"], o, d["dout"], lse, bias, land, dq, dk, dv, dbias,
                              ws, stream)
            ev[5].record(stream)
        torch.cuda.synchronize()
        if r >= warmup:
            fwd_t.append(ev[0].elapsed_time(ev[1]) * 1e3)
            if backward:
                bwd_t.append(ev[2].elapsed_time(ev[3]) * 1e3)
            if with_o:
                bwdo_t.append(ev[4].elapsed_time(ev[5]) * 1e3)
    assert C.swin_attn_status(attn.plan) == 0
    tokens = wl.batch * wl.tokens
    fwd_us = statistics.median(fwd_t)
    f_roof = roof_us(fwd_flop, fwd_bytes, peaks)
    res = {"kernels": {1: "simt", 2: "tcgen05"}[attn.info.impl], "tokens": tokens, "reps": reps, "warmup": warmup,
           "l2": "1 GiB written before every launch", "timing": "median of CUDA-event launch times",
           "fwd": {"us": fwd_us, "us_min": min(fwd_t), "mtok_s": tokens / fwd_us, "tflops": fwd_flop / fwd_us / 1e6,
                   "roof_us": f_roof, "roof_frac": f_roof / fwd_us, "alg_bytes": fwd_bytes,
                   "lse_written": bool(wl.backward)}}
    if backward:
        bwd_us = statistics.median(bwd_t)
        b_roof = roof_us(bwd_flop, bwd_bytes, peaks)
        res["bwd"] = {"us": bwd_us, "us_min": min(bwd_t), "tflops": bwd_flop / bwd_us / 1e6, "roof_us": b_roof,
                      "roof_frac": b_roof / bwd_us, "alg_bytes": bwd_bytes,
                      "roof_frac_moved": roof_us(bwd_flop, bwd_moved, peaks) / bwd_us, "alg_bytes_moved": bwd_moved}
        res["fwd_bwd_mtok_s"] = tokens / (fwd_us + bwd_us)
        if with_o:
            us = statistics.median(bwdo_t)
            res["bwd_o"] = {"us": us, "tflops": bwd_flop / us / 1e6, "roof_us": b_roof, "roof_frac": b_roof / us,
                            "api": "swin_attn_bwd_o: delta = dO . O from the forward's bf16 output"}
    elif wl.backward:
        res["bwd"] = "no backward kernel for this configuration yet"
    tgt = TARGETS.get(wl.name)
    res["target"] = tgt
    if tgt:
        res["meets_target"] = all(res[k_]["roof_frac"] >= v for k_, v in tgt.items())
    if wl.name in NOTES:
        res["note"] = NOTES[wl.name]
    del attn
    return res


def time_pair(wl, peaks, flush, reps=50, warmup=10):
    """The W-MSA + SW-MSA block pair on one grid (shift 0, then floor(w/2)),
    two plans built once: the forward of both layers back to back, then the
    backward of both (second layer first), each pair of launches timed as one
    region after an L2 flush; medians over `reps`. Roofline: the sum of both
    layers' roofline times over the measured time."""
    import torch
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300 import workloads
    from shifted_window_attention_cyclic_gb300.functional import SwinBlockPair
    dev = torch.device("cuda", torch.cuda.current_device())
    pair = SwinBlockPair(wl.grid, wl.window, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.dtype, wl.has_land)
    layers = [workloads.custom(wl.grid, wl.window, sh, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.dtype,
                               wl.land_p, seed_index=wl.index + 40 + i, name=wl.name + ("_wmsa", "_swmsa")[i])
              for i, sh in enumerate(((0,) * len(wl.grid), pair.shift))]
    xs = [workloads.generate(lw) for lw in layers]
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    t = [{k_: torch.from_numpy(x[k_]).to(dev).to(tdt) for k_ in ("q", "k", "v", "dout")} for x in xs]
    for x, d in zip(xs, t):
        d["bias"] = torch.from_numpy(x["bias"]).to(dev)
    land = torch.from_numpy(xs[0]["land"]).to(dev) if xs[0]["land"] is not None else None
    first = (t[0]["q"], t[0]["k"], t[0]["v"], t[0]["bias"])
    second = (t[1]["q"], t[1]["k"], t[1]["v"], t[1]["bias"])
    fwd_t, bwd_t = [], []
    stream = torch.cuda.current_stream()
    for r in range(warmup + reps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        flush.add_(1)
        ev[0].record(stream)
        (o1, l1), (o2, l2) = pair.forward(first, second, land)
        ev[1].record(stream)
        flush.add_(1)
        ev[2].record(stream)
        pair.backward(first, second, t[0]["dout"], t[1]["dout"], l1, l2, land)
        ev[3].record(stream)
        torch.cuda.synchronize()
        if r >= warmup:
            fwd_t.append(ev[0].elapsed_time(ev[1]) * 1e3)
            bwd_t.append(ev[2].elapsed_time(ev[3]) * 1e3)
    assert C.swin_attn_status(pair.wmsa.plan) == 0 and C.swin_attn_status(pair.swmsa.plan) == 0
    f_roof = b_roof = 0.0
    for lw, x, attn in zip(layers, xs, (pair.wmsa, pair.swmsa)):
        win_src = C.swin_attn_plan_tables(attn.plan)[0]
        ff, bf, fb, bb, _ = workload_counts(lw, win_src, x["land"])
        f_roof += roof_us(ff, fb, peaks)
        b_roof += roof_us(bf, bb, peaks)
    tokens = wl.batch * wl.tokens
    fwd_us, bwd_us = statistics.median(fwd_t), statistics.median(bwd_t)
    return {"grid": list(wl.grid), "window": list(wl.window), "shifts": [[0] * len(wl.grid), list(pair.shift)],
            "plans": "two, built once and reused (the shift changes the routing tables)",
            "l2": "1 GiB written before each pair of launches", "reps": reps, "warmup": warmup,
            "fwd": {"us": fwd_us, "mtok_s": tokens / fwd_us, "roof_us": f_roof, "roof_frac": f_roof / fwd_us},
            "bwd": {"us": bwd_us, "roof_us": b_roof, "roof_frac": b_roof / bwd_us},
            "fwd_bwd_mtok_s": tokens / (fwd_us + bwd_us)}


def block_counts(wl, win_src, land):
    """Algorithmic FLOPs and bytes of the attention half of a Swin block in one
    launch: LayerNorm + QKV projection (2 N C 3C), the window attention (the
    forward's 4 B sum n^2 C) and the out-projection (2 N C C); bytes: x in and
    y out (2 N C e), the weights (4 C^2 e) and the LayerNorm and bias vectors,
    land and the bias table. Q, K, V and O stay on chip, so they cost nothing."""
    fwd_flop, _, _, _, _ = workload_counts(wl, win_src, land, lse_written=False)
    N, C, e = wl.batch * wl.tokens, wl.channels, 2
    rows = int(np.prod([2 * w - 1 for w in wl.window]))
    flop = 2.0 * N * C * 3 * C + fwd_flop + 2.0 * N * C * C
    nbytes = 2 * N * C * e + 4 * C * C * e + 4 * (6 * C) + (N if land is not None else 0) + rows * wl.heads * 4
    return flop, nbytes


def time_block(wl, peaks, flush, reps=50, warmup=10):
    """The attention half of a Swin block (LayerNorm + QKV projection, SW-MSA,
    out-projection + residual) in one launch of swin_attn_block_fwd, timed
    launch by launch after an L2 flush (medians over `reps`); beside it, for
    context, the same block unfused: torch layer_norm and linear (cuBLAS)
    around this library's attention forward, timed as one region."""
    import torch
    import torch.nn.functional as F
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300 import workloads
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    dev = torch.device("cuda", torch.cuda.current_device())
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, "bf16",
                               wl.has_land)
    h = workloads.generate_block(wl)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf = lambda a: f32(a).to(torch.bfloat16)
    x, w_qkv, w_o = bf(h["x"]), bf(h["w_qkv"]), bf(h["w_o"])
    gamma, beta, b_qkv, b_o, bias = f32(h["gamma"]), f32(h["beta"]), f32(h["b_qkv"]), f32(h["b_o"]), f32(h["bias"])
    land = f32(h["land"]) if h["land"] is not None else None
    y = torch.empty_like(x)
    c = wl.channels

    def unfused():
        xn = F.layer_norm(x, (c,), gamma.to(torch.bfloat16), beta.to(torch.bfloat16), 1e-5)
        q, k, v = (t.contiguous() for t in F.linear(xn, w_qkv, b_qkv.to(torch.bfloat16)).split(c, dim=-1))
        o, _ = attn.forward(q, k, v, bias, land, need_lse=False)
        return x + F.linear(o, w_o, b_o.to(torch.bfloat16))

    stream = torch.cuda.current_stream()
    times = {"fused": [], "unfused": []}
    for r in range(warmup + reps):
        for key in times:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            flush.add_(1)
            ev[0].record(stream)
            if key == "fused":
                attn.block_forward(x, gamma, beta, w_qkv, b_qkv, w_o, b_o, bias, land, 1e-5, y=y)
            else:
                unfused()
            ev[1].record(stream)
            torch.cuda.synchronize()
            if r >= warmup:
                times[key].append(ev[0].elapsed_time(ev[1]) * 1e3)
    assert C.swin_attn_status(attn.plan) == 0
    win_src = C.swin_attn_plan_tables(attn.plan)[0]
    flop, nbytes = block_counts(wl, win_src, h["land"])
    fused_us, unfused_us = statistics.median(times["fused"]), statistics.median(times["unfused"])
    roof = roof_us(flop, nbytes, peaks)
    tokens = wl.batch * wl.tokens
    return {"grid": list(wl.grid), "window": list(wl.window), "channels": c,
            "l2": "1 GiB written before each launch", "reps": reps, "warmup": warmup,
            "fwd": {"us": fused_us, "mtok_s": tokens / fused_us, "roof_us": roof, "roof_frac": roof / fused_us,
                    "tflops": flop / fused_us / 1e6, "bound": "tensor" if flop / (peaks["bf16_tflops"] * 1e12) >
                    nbytes / (peaks["hbm_gbs"] * 1e9) else "hbm"},
            "unfused_us": unfused_us,
            "unfused": "torch layer_norm + linear (cuBLAS) around swin_attn_fwd, for context"}


KERNEL_UNITS = {"tcgen05": "swin_tc.cu", "simt": "swin_simt.cu"}


def kernel_source_hash(kernels="tcgen05"):
    """Hash of the CUDA sources a kernel family compiles from: its translation
    unit (swin_tc.cu or swin_simt.cu), the launch plans (swin_api.cu), and the
    headers either includes, followed transitively. Changes to other kernels
    (the head_dim-128 ones) leave it alone."""
    csrc = os.path.join(ROOT, "shifted_window_attention_cyclic_gb300", "csrc")
    todo = [os.path.join(csrc, KERNEL_UNITS[kernels]), os.path.join(csrc, "swin_api.cu")]
    seen = []
    while todo:
        path = os.path.normpath(todo.pop(0))
        if path in seen or not os.path.exists(path):
            continue
        seen.append(path)
        with open(path) as f:
            for line in f:
                line = line.strip()
                if line.startswith('#include "'):
                    todo.append(os.path.join(os.path.dirname(path), line.split('"')[1]))
    h = hashlib.sha256()
    for path in sorted(seen):
        with open(path, "rb") as f:
            h.update(os.path.relpath(path, ROOT).encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_hash, workload, kernels, path=None):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, only if it was captured from the current kernel sources, for
    this workload and this kernel family; None otherwise."""
    path = path or os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    if (t.get("kernel_source_hash") != kernel_hash or t.get("workload") != workload
            or t.get("kernels") != kernels):
        return None
    return t.get("bwd_dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[4:8]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x, device):
    """The largest x of all ranks (x itself when the job has one rank): each
    rank times its own replica, and the job is as slow as its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, tokens_per_rank, ms_per_step):
    """Whole-job throughput in Mtokens/s: every rank processes its own batch."""
    return world * tokens_per_rank / (ms_per_step * 1e-3) / 1e6


def oracle_sample_rate(wl, x, windows, seed=0):
    """Time the oracle (fwd + bwd, fp64) on `windows` windows; returns (tokens, seconds)."""
    import oracle
    pb = oracle.Problem(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.has_land)
    rng = np.random.default_rng(seed)
    population = wl.batch * pb.nwin
    ids = rng.choice(population, size=windows, replace=windows > population)  # small grids repeat windows
    win_src = oracle.tables(pb)[0]
    tokens = int(sum((win_src[i % pb.nwin] >= 0).sum() for i in ids))
    t0 = time.perf_counter()
    oracle.fwd_windows(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], win_ids=ids)
    oracle.bwd_windows(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"], win_ids=ids)
    return tokens, time.perf_counter() - t0


PARITY_BAR = {"bf16": {"rel_l2": 5e-3, "max_abs": 2e-2}, "f32": {"rel_l2": None, "max_abs": 1e-5}}


def parity_sample(wl, x, outs, windows=512, seed=7):
    """Part of the cpu_baseline leg: the oracle against this run's own device
    results (the timed launch configuration, full size, same inputs) on a
    sample of windows, namely the corner, seam and ragged-edge windows of
    each dimension plus random ones. Returns max-abs and rel-L2 of O, dQ, dK
    and dV over the sampled windows' real slots, and whether they meet the bar."""
    import itertools
    import torch
    import oracle
    pb = oracle.Problem(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.has_land)
    nwd = pb.windows_per_dim
    edge = {int(np.ravel_multi_index(c, nwd))
            for c in itertools.product(*[sorted({0, 1, n // 2, n - 2, n - 1} & set(range(n))) for n in nwd])}
    rng = np.random.default_rng(seed)
    total = wl.batch * pb.nwin
    rand = rng.choice(total, size=min(windows, total), replace=False)
    ids = np.array(sorted(set(rand.tolist()) | {b * pb.nwin + w for b in range(wl.batch) for w in edge}), np.int64)
    win_src = oracle.tables(pb)[0]
    o_ref, _ = oracle.fwd_windows(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], win_ids=ids)
    g_ref = oracle.bwd_windows(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"], win_ids=ids,
                               want=("dq", "dk", "dv"))
    src = win_src[ids % pb.nwin]
    valid = src >= 0
    rows = ((ids // pb.nwin)[:, None] * pb.tokens + np.maximum(src, 0))[valid]
    res = {}
    bar = PARITY_BAR[wl.dtype]
    ok = True
    for key, ref in (("o", o_ref), ("dq", g_ref["dq"]), ("dk", g_ref["dk"]), ("dv", g_ref["dv"])):
        dev = outs[key].reshape(-1, pb.channels)
        got = dev[torch.from_numpy(rows).to(dev.device)].double().cpu().numpy()
        r = np.asarray(ref, np.float64)[valid]
        err = got - r
        max_abs = float(np.abs(err).max())
        rel_l2 = float(np.linalg.norm(err) / max(np.linalg.norm(r), 1e-300))
        res[key] = {"max_abs": max_abs, "rel_l2": rel_l2}
        ok &= max_abs <= bar["max_abs"] and (bar["rel_l2"] is None or rel_l2 <= bar["rel_l2"])
    res["bar"] = bar
    res["within_bar"] = bool(ok)
    res["sample"] = "%d windows (corner, seam, ragged edges and random), %d tokens, fp64 C oracle" % (
        len(ids), int(valid.sum()))
    return res


def cpu_baseline(wl, x, target_s=15.0, target_1core_s=10.0):
    """The oracle as it stands, timed on this host's cores over a bounded
    sample of windows (fwd + bwd): once with every core (OpenMP default) and
    once single-threaded (a child process with OMP_NUM_THREADS=1)."""
    import oracle
    oracle.build()
    calib = 256
    tok, dt = oracle_sample_rate(wl, x, calib, seed=1)
    per_window = dt / calib
    nwin = oracle.Problem(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim).nwin
    windows = int(max(calib, min(max(wl.batch * nwin, 4096), target_s / max(per_window, 1e-6))))
    tok, dt = oracle_sample_rate(wl, x, windows, seed=2)
    cores = oracle.num_threads()
    res = {"value": tok / dt / 1e6, "unit": "Mtokens/s", "cores": cores, "kind": "oracle",
           "sample": "%d random windows of %s (%d tokens), fwd+bwd, fp64 C oracle, %.1f s" %
                     (windows, wl.name, tok, dt)}
    w1 = int(max(8, min(windows, target_1core_s / max(per_window * cores, 1e-6))))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", str(w1), "--workload", wl.name],
                       capture_output=True, text=True, env=env, timeout=600)
    try:
        one = json.loads(r.stdout.strip().splitlines()[-1])
        res["single_core"] = {"value": one["tokens"] / one["seconds"] / 1e6, "unit": "Mtokens/s",
                              "cores": one["cores"],
                              "sample": "%d random windows (%d tokens), %.1f s" % (w1, one["tokens"], one["seconds"])}
    except (IndexError, ValueError, KeyError):
        res["single_core"] = {"error": (r.stderr or r.stdout)[-300:]}
    return res


def oracle_sample_main(windows, wl):
    """Child process of cpu_baseline: time the oracle on `windows` windows with
    the thread count its environment sets, print one JSON line."""
    from shifted_window_attention_cyclic_gb300 import workloads
    import oracle
    oracle.build()
    x = workloads.generate(wl)
    tok, dt = oracle_sample_rate(wl, x, windows, seed=4)
    print(json.dumps({"tokens": tok, "seconds": dt, "cores": oracle.num_threads()}))
    return 0


def run_reference(args, wl):
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    from shifted_window_attention_cyclic_gb300 import workloads
    import oracle
    oracle.build()
    x = workloads.generate(wl)
    # size each step so that the whole run stays within ~2 minutes of CPU time
    tok, dt = oracle_sample_rate(wl, x, 8, seed=3)
    per_window = dt / 8
    budget = 120.0 / max(1, args.steps + args.warmup)
    windows = int(max(1, min(512, budget / max(per_window, 1e-6))))
    for s in range(args.warmup):
        oracle_sample_rate(wl, x, windows, seed=100 + s)
    total_tok, total_t = 0, 0.0
    for s in range(args.steps):
        tok, dt = oracle_sample_rate(wl, x, windows, seed=1000 + s)
        total_tok += tok
        total_t += dt
    value = total_tok / total_t / 1e6
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "Mtokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, shapes of the pages' workloads)",
            "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": "Mtokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": "%d random windows per step of %s, fwd+bwd, fp64 C oracle" %
                                       (windows, wl.name)},
            "e2e": {"value": value, "unit": "Mtokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def config_of(wl):
    tensor_mb = wl.batch * wl.tokens * wl.channels * (2 if wl.dtype == "bf16" else 4) / 1e6
    return {"workload": "%s: B=%d grid %s C=%d heads %dx%d window %s shift %s periodic %s land p %s %s" %
                        (wl.name, wl.batch, "x".join(map(str, wl.grid)), wl.channels, wl.heads, wl.head_dim,
                         "x".join(map(str, wl.window)), tuple(wl.shift), tuple(wl.periodic), wl.land_p, wl.dtype)
                        + ("" if wl.bias else " no bias"),
            "global_batch": wl.batch, "tokens_per_batch": wl.batch * wl.tokens,
            "parallelism": "replicas (independent problem per GPU)",
            "l2": ("inputs larger than L2 (each tensor %.0f MB > 129 MB), no flush" if tensor_mb > 129 else
                   "inputs smaller than L2 (each tensor %.0f MB), no flush: L2-resident timing") % tensor_mb}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernels", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config table (all five workloads)")
    ap.add_argument("--config-reps", type=int, default=50)
    ap.add_argument("--only-block", action="store_true",
                    help="time only the fused block (LayerNorm + QKV, SW-MSA, out-projection) on --workload")
    ap.add_argument("--oracle-sample", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    from shifted_window_attention_cyclic_gb300 import workloads
    wl = workloads.WORKLOADS[args.workload]
    if args.oracle_sample:
        return oracle_sample_main(args.oracle_sample, wl)
    if args.impl == "reference":
        return run_reference(args, wl)
    if args.only_block:
        import torch
        peaks, _ = load_peaks()
        flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        print(json.dumps({"workload": wl.name, "block_fused": time_block(wl, peaks, flush, reps=args.steps,
                                                                         warmup=args.warmup)}))
        return 0

    import torch
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__
    __graft_entry__.build_library()
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention

    x = workloads.generate(wl)
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch,
                               wl.dtype, wl.has_land, args.kernels)
    win_src = C.swin_attn_plan_tables(attn.plan)[0]
    fwd_flop, bwd_flop, fwd_bytes, bwd_bytes, bwd_moved = workload_counts(wl, win_src, x["land"])
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    host = {k_: torch.from_numpy(x[k_]).to(tdt).pin_memory() for k_ in ("q", "k", "v", "dout")}
    if wl.bias:  # a workload without a relative-position bias passes NULL bias and dbias
        host["bias"] = torch.from_numpy(x["bias"]).pin_memory()
    if x["land"] is not None:
        host["land"] = torch.from_numpy(x["land"]).pin_memory()
    d = {k_: t.to(dev) for k_, t in host.items()}
    d_land = d.get("land")
    o = torch.empty(attn.shape, dtype=tdt, device=dev)
    lse = torch.empty(attn.lse_shape, dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty(attn.shape, dtype=tdt, device=dev) for _ in range(3))
    dbias = attn.new_bias() if wl.bias else None
    ws = attn.workspace()
    stream = torch.cuda.current_stream()

    outs = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    if dbias is not None:
        outs["dbias"] = dbias

    def step(src=None, out=None):
        src = d if src is None else src
        r = outs if out is None else out
        land_ = src.get("land")
        C.swin_attn_fwd(attn.plan, src["q"], src["k"], src["v"], src.get("bias"), land_, r["o"], r["lse"], stream)
        C.swin_attn_bwd(attn.plan, src["q"], src["k"], src["v"], src["dout"], r["lse"], src.get("bias"), land_,
                        r["dq"], r["dk"], r["dv"], r.get("dbias"), ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == 0

    # timed region: K steps, events per launch on the launching stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for e0, e1, e2 in ev:
        e0.record(stream)
        C.swin_attn_fwd(attn.plan, d["q"], d["k"], d["v"], d.get("bias"), d_land, o, lse, stream)
        e1.record(stream)
        C.swin_attn_bwd(attn.plan, d["q"], d["k"], d["v"], d["dout"], lse, d.get("bias"), d_land, dq, dk, dv, dbias,
                        ws, stream)
        e2.record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    assert C.swin_attn_status(attn.plan) == 0
    total_ms = start.elapsed_time(end)
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    tokens = wl.batch * wl.tokens
    value = job_rate(world, tokens, ms_per_step)
    fwd_avg = statistics.median(fwd_ms)  # per-launch breakdown: medians of the K steps
    bwd_avg = statistics.median(bwd_ms)
    peaks, peak_kind = load_peaks()
    hbm = peaks["hbm_gbs"]
    fwd_roof_us = roof_us(fwd_flop, fwd_bytes, peaks)
    bwd_roof_us = roof_us(bwd_flop, bwd_bytes, peaks)
    bwd_gbs = bwd_bytes / (bwd_avg * 1e-3) / 1e9
    khash = kernel_source_hash({1: "simt", 2: "tcgen05"}[attn.info.impl])

    # end to end through the public API with host buffers: H2D inputs, fwd, bwd, D2H results
    host_out = {k_: torch.empty(attn.shape, dtype=tdt).pin_memory() for k_ in ("o", "dq", "dk", "dv")}
    if dbias is not None:
        host_out["dbias"] = torch.empty_like(dbias, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    # Every step copies its inputs host->device and its results device->host
    # inside the timed region. As in a training input pipeline, the copies
    # run on two more streams and both device sets (inputs, results) are
    # double-buffered: step k+1's inputs come in and step k-1's results go
    # out while step k computes (the two copy directions overlap).
    in_stream, out_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    dsets = [d, {k_: torch.empty_like(t) for k_, t in d.items()}]
    osets = [outs, {k_: torch.empty_like(t) for k_, t in outs.items()}]
    in_ready, in_free, out_ready, out_free = ([torch.cuda.Event(), torch.cuda.Event()] for _ in range(4))

    def h2d_copy(j):
        with torch.cuda.stream(in_stream):
            in_stream.wait_event(in_free[j])
            for k_, t in host.items():
                dsets[j][k_].copy_(t, non_blocking=True)
            in_ready[j].record(in_stream)

    def compute(j):
        stream.wait_event(in_ready[j])
        stream.wait_event(out_free[j])
        step(dsets[j], osets[j])
        in_free[j].record(stream)
        out_ready[j].record(stream)

    def d2h_copy(j):
        with torch.cuda.stream(out_stream):
            out_stream.wait_event(out_ready[j])
            for k_ in host_out:
                host_out[k_].copy_(osets[j][k_], non_blocking=True)
            out_free[j].record(out_stream)

    def e2e_run(steps):
        start = torch.cuda.Event()
        start.record(stream)
        in_stream.wait_event(start)
        out_stream.wait_event(start)
        h2d_copy(0)
        for k_ in range(steps):
            if k_ + 1 < steps:
                h2d_copy((k_ + 1) % 2)
            compute(k_ % 2)
            d2h_copy(k_ % 2)
        done = torch.cuda.Event()
        done.record(out_stream)
        stream.wait_event(done)  # the timed region ends after the last result copy

    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dev)

    # every workload, launch by launch, L2 flushed before each launch
    configs = None
    if rank == 0 and not args.no_configs:
        flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        flush.zero_()
        csampler = ClockSampler(dev.index)
        csampler.start()
        configs = {}
        for name in list(TARGETS) + EXTRA:
            cwl = workloads.WORKLOADS[name]
            cx = x if name == wl.name else workloads.generate(cwl)
            reps, warm = EXTRA_REPS.get(name, (args.config_reps, 10))
            configs[name] = time_config(cwl, cx, peaks, flush, reps=min(reps, args.config_reps), warmup=warm)
            configs[name]["config"] = config_of(cwl)["workload"]
        # the W-MSA + SW-MSA pair on the eddy-resolving ocean grid (TERRA's Wenhai stand-in)
        configs["block_pair_eddy_ocean"] = time_pair(workloads.WORKLOADS["eddy_ocean"], peaks, flush,
                                                     reps=args.config_reps, warmup=10)
        # the attention half of a Swin block in one launch (LayerNorm + QKV, SW-MSA, out-projection)
        for name in ("depth3d", "grid1deg"):
            configs["block_fused_" + name] = time_block(workloads.WORKLOADS[name], peaks, flush,
                                                        reps=args.config_reps, warmup=10)
        configs["clocks"] = csampler.stop()
        configs["peaks"] = {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                            "source": peak_kind, "which": "burst bf16 peak, measured copy bandwidth"}
        del flush
        torch.cuda.empty_cache()

    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and int(np.prod(wl.window)) > ORACLE_WINDOW_SLOTS:
        why = ("windows of %d slots: the per-window oracle holds n x n fp64 matrices per thread; parity at this "
               "size is tests/test_gpu_large_windows_sampled.py (the oracle's sampled rows)" % int(np.prod(wl.window)))
        cpu, parity = {"skipped": why}, {"skipped": why}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, x)
        try:  # a report only: its failure must not cost the measurement
            parity = parity_sample(wl, x, outs)
        except Exception as e:  # noqa: BLE001
            parity = {"error": repr(e)}

    if rank == 0:
        kernels = {1: "simt", 2: "tcgen05"}[attn.info.impl]
        line = {
            "metric": METRIC, "value": value, "unit": "Mtokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded, shapes of the pages' workloads)",
            "config": config_of(wl),
            "fwd": {"mtok_s": tokens / (fwd_avg * 1e-3) / 1e6, "us": fwd_avg * 1e3, "roof_us": fwd_roof_us,
                    "roof_frac": fwd_roof_us / (fwd_avg * 1e3), "tflops": fwd_flop / (fwd_avg * 1e-3) / 1e12,
                    "alg_bytes": fwd_bytes},
            "bwd": {"us": bwd_avg * 1e3, "roof_us": bwd_roof_us, "roof_frac": bwd_roof_us / (bwd_avg * 1e3),
                    "tflops": bwd_flop / (bwd_avg * 1e-3) / 1e12, "alg_bytes": bwd_bytes,
                    "alg_bytes_moved": bwd_moved,
                    "roof_frac_moved": roof_us(bwd_flop, bwd_moved, peaks) / (bwd_avg * 1e3)},
            "fwd_bwd": {"mtok_s": value / world, "roof_frac": (fwd_roof_us + bwd_roof_us) / (ms_per_step * 1e3)},
            "roofline": {"bound": "hbm", "kernel": "swin_attn_bwd (main kernel + dBias fold)",
                         "achieved": bwd_gbs, "peak": hbm, "unit": "GB/s", "frac": bwd_gbs / hbm,
                         "peak_source": peak_kind + " (copy bandwidth, burst)",
                         "traffic": profiled_traffic(khash, args.workload, kernels),
                         "alg_bytes_per_launch": bwd_bytes,
                         "alg_bytes_note": "Q, K, V, O, dO, dQ, dK, dV + LSE, delta, land, bias, dBias; this "
                                           "backward reads neither O nor delta: it moves alg_bytes_moved",
                         "frac_moved": bwd_moved / (bwd_avg * 1e-3) / 1e9 / hbm},
            "configs": configs,
            "clocks": clocks,
            "e2e": {"value": job_rate(world, tokens, e2e_ms), "unit": "Mtokens/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": 3 * args.steps,
            "impl_kernels": kernels,
            "kernel_source_hash": khash,
            "cpu_baseline": cpu,
            "parity": parity,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
