#!/usr/bin/env python
"""Benchmark of the FP8 up-projection training step on GB300.

Workload (GPT-2-small-shaped MLP up-projection): x [8192 x 768] ~ N(0,1) with 0.1 % of
the entries x100, W [768 x 3072] ~ N(0, 0.02), dy [8192 x 3072] log-normal (median 1e-4,
sigma_log 2, random sign). One step = one pass of the whole hot path with per-tensor
delayed scaling (amax history of 16):
  requantise W (amax, scale, E4M3 cast into W_q [K,N] and W_q^T [N,K])
  quantise x (E4M3, x_q and x_q^T)          forward GEMM  y  = x W         (tcgen05)
  quantise dy (E5M2, dy_q and dy_q^T)       dgrad GEMM    dx = dy W^T
                                            wgrad GEMM    dW = x^T dy
  push the x, W and dy amaxes into their histories.
The step is captured into a CUDA graph; each timed step replays it with CUDA events around
the launch, after writing a 256 MiB buffer to flush the 129 MB L2 (not timed). Per-kernel
times come from the same stages launched eagerly in the same loop, each behind a flush. value = the step's GEMM FLOPs (3 x 2MNK) over the
measured step time, summed over ranks (each rank its own batch: weak scaling).

--impl reference times the CPU oracle (test infrastructure) on a bounded sample of the
same step on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 up-proj GEMM TFLOP/s (% FP8 peak); quantize-cast GB/s (% HBM)"
M, K, N = 8192, 768, 3072
HIST = 16
FLUSH_BYTES = 256 << 20
# Roofline denominators: HBM copy GB/s and dense bf16 TFLOP/s (burst) from MEASURED_PEAKS.json,
# else these earlier GB300 measurements; the FP8 dense peak is the bf16 figure times the
# nominal fp8/bf16 ratio 4.5 / 2.25 = 2.
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return FALLBACK_PEAKS["hbm_gbs"], FALLBACK_PEAKS["bf16_tflops"], "fallback"


def env_rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


# --------------------------------------------------------------------------------------
# clocks sampler
# --------------------------------------------------------------------------------------
class Clocks:
    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------
# The sources that decide each stage's kernel and launch (kernel body, its headers, the
# host code that picks and launches it): a stage's DRAM counters stay valid while these hash
# the same as when the counters were taken.
_CAST_SOURCES = ("quant.cu", "cast.cuh", "ptx.cuh", "kernels.h", "api.cu")
_GEMM_SOURCES = ("gemm.cu", "cast.cuh", "ptx.cuh", "kernels.h", "api.cu")
STAGE_SOURCES = {"requant_w": _CAST_SOURCES, "quant_x": _CAST_SOURCES, "quant_dy": _CAST_SOURCES,
                 "gemm_fwd": _GEMM_SOURCES, "gemm_bwd": _GEMM_SOURCES}


def traffic_table():
    """Per-launch DRAM bytes from the committed ncu summary, keyed by stage, valid only
    while the stage's kernel sources hash the same as when the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic_per_launch.txt")
    out = {}
    if not os.path.exists(path):
        return out
    for line in open(path):
        line = line.split("#")[0].split()
        if len(line) == 3 and line[0] in STAGE_SOURCES and line[2] == source_hash(STAGE_SOURCES[line[0]]):
            out[line[0]] = float(line[1])
    return out


def source_hash(files, read=None):
    """First 16 hex digits of the SHA-256 of the named csrc files, in order. `read` maps a
    file name to its bytes (default: the working tree)."""
    d = os.path.join(ROOT, "fp8_mixed_precision_saturating_gb300", "csrc")
    read = read or (lambda f: open(os.path.join(d, f), "rb").read())
    hsh = hashlib.sha256()
    for f in files:
        hsh.update(f.encode() + b"\0")
        hsh.update(read(f))
    return hsh.hexdigest()[:16]


def rank_seeds(rank: int):
    """Seeds of rank r's own batch (x, dy): rank 0 uses the workload's seeds."""
    return (1000 * 2 + 0, 2002) if rank == 0 else (2000 + 10 * rank, 2002 + 10 * rank)


def max_over_ranks(total_ms: float, world: int, device) -> float:
    """The slowest rank's timed total (every rank calls this)."""
    if world <= 1:
        return total_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(step_flops: float, steps: int, world: int, total_ms: float) -> float:
    """TFLOP/s of the whole job: every rank ran `steps` steps of its own batch."""
    return step_flops * steps * world / (total_ms * 1e-3) / 1e12


def run_gpu(args):
    import numpy as np
    import torch

    rank, local_rank, world = env_rank()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    import fp8_mixed_precision_saturating_gb300 as g
    from datagen import workload_inputs, lognormal_grad_bf16, outlier_normal_bf16

    w = workload_inputs("gpt2s_upproj_fwd")
    sx, sdy = rank_seeds(rank)
    x_h = w["x"] if rank == 0 else outlier_normal_bf16(sx, (M, K))
    w_h = w["w"]
    dy_h = lognormal_grad_bf16(sdy, (M, N))

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    x, wm, dy = dev(x_h), dev(w_h), dev(dy_h)
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device="cuda")
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    wst, xst, gst = g.TensorState(HIST), g.TensorState(HIST), g.TensorState(HIST)
    wq, wqT, xq, xqT, dyq, dyqT = u8(K, N), u8(N, K), u8(M, K), u8(K, M), u8(M, N), u8(N, M)
    y, dx, dw = bf(M, N), bf(M, K), bf(K, N)
    D = g.FP8_SCALE_DELAYED
    T = g.FP8_GRAN_TENSOR
    gemm_flops = 2.0 * M * N * K

    # the backward's two GEMMs run as one grouped launch (wgrad split over its tokens through
    # the workspace, dgrad beside it); the forward GEMM gets the same workspace (unused: its
    # 384 tiles fill the GPU)
    bwd = [g.mm_problem(xqT, 0, dyqT, 1, K, N, M, M, M, xst.scale_inv, gst.scale_inv, dw, N),
           g.mm_problem(dyq, 1, wq, 0, M, K, N, N, N, gst.scale_inv, wst.scale_inv, dx, K)]
    ws_bytes = max(g.fp8_scaled_mm_grouped_workspace_bytes(bwd), g.fp8_scaled_mm_workspace_bytes(M, N, K))
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    # (name, call, kernels launched, algorithmic flops, algorithmic bytes)
    stages = [
        ("requant_w", lambda: g.fp8_requantize_weights(wm, K, N, T, D, wst, wq, wqT), 1, 0.0, K * N * 4.0),
        ("quant_x", lambda: g.fp8_quantize(x, M, K, K, g.FP8_E4M3, T, D, xst, xq, xqT), 1, 0.0, M * K * 4.0),
        ("gemm_fwd", lambda: g.fp8_scaled_mm_ws(xq, 0, wqT, 0, M, N, K, K, K, T, xst.scale_inv, wst.scale_inv, y, N,
                                                ws, ws_bytes), 1, gemm_flops, 0.0),
        ("quant_dy", lambda: g.fp8_quantize(dy, M, N, N, g.FP8_E5M2, T, D, gst, dyq, dyqT), 1, 0.0, M * N * 4.0),
        ("gemm_bwd", lambda: g.fp8_scaled_mm_grouped(bwd, ws, ws_bytes), 1, 2 * gemm_flops, 0.0),
        ("commit", lambda: g.fp8_history_commit_many([wst, xst, gst]), 1, 0.0, 0.0),
    ]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _, fn, *_ in stages:  # eager pass: sets kernel attributes and caches
            fn()
        torch.cuda.synchronize()
        # the step is one CUDA graph, replayed once per timed step with CUDA events around the
        # launch (the graph launch itself counts). Per-kernel times come from the same stages
        # launched eagerly in the same loop, each behind an L2 flush: the GPU is still busy
        # with the flush while the host enqueues the stage, so the events bracket only the
        # kernel (cold L2, no event nodes inside a graph).
        # the step's dependency graph: W's refresh beside x's cast on two streams (measured
        # 2 us faster per step than the one-launch fp8_quantize_many of both), then the
        # forward GEMM, dy's cast, the grouped backward GEMMs and the history commit
        side = torch.cuda.Stream()
        fn = {name: f for name, f, *_ in stages}
        plain = torch.cuda.CUDAGraph()
        with torch.cuda.graph(plain, stream=stream):
            side.wait_stream(stream)
            fn["requant_w"]()
            with torch.cuda.stream(side):
                fn["quant_x"]()
            stream.wait_stream(side)
            fn["gemm_fwd"]()
            fn["quant_dy"]()
            fn["gemm_bwd"]()
            fn["commit"]()
        for st in (wst, xst, gst):
            st.reset()  # the delayed-scaling state starts empty (bootstrap step first)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in stages]

        def step():
            flush.zero_()  # L2 flush, outside the timed events
            e0.record(stream)
            plain.replay()
            e1.record(stream)
            for (a, b), (_, fn, *_) in zip(ev, stages):
                flush.zero_()
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1), [a.elapsed_time(b) for a, b in ev]

        for _ in range(args.warmup):
            step()
        clocks = Clocks(local_rank)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        clocks.start()
        time.sleep(0.3)  # let the sampler see the first samples
        wall0 = time.perf_counter()
        per_step = [step() for _ in range(args.steps)]
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if world > 1:
            torch.distributed.barrier()
        clk = clocks.stop()
        g.fp8_poll_device_error()

    step_ms = [t for t, _ in per_step]
    stage_ms = [sum(t[i] for _, t in per_step) / args.steps for i in range(len(stages))]
    probe_step_ms = sum(stage_ms)
    total_ms = max_over_ranks(sum(step_ms), world, "cuda")
    step_flops = sum(s[3] for s in stages)
    value = weak_scaling_value(step_flops, args.steps, world, total_ms)

    hbm, bf16_tf, peak_src = load_peaks()
    fp8_peak = bf16_tf * 2.0
    traffic = traffic_table()
    kernels = {}
    for (name, _, nk, fl, by), ms in zip(stages, stage_ms):
        kd = {"ms": round(ms, 5), "launches": nk}
        if fl:
            kd.update(achieved=round(fl / (ms * 1e-3) / 1e12, 1), unit="TFLOP/s", frac=round(fl / (ms * 1e-3) / 1e12 / fp8_peak, 4))
        elif by:
            kd.update(achieved=round(by / (ms * 1e-3) / 1e9, 1), unit="GB/s", frac=round(by / (ms * 1e-3) / 1e9 / hbm, 4))
        kernels[name] = kd
    dom_i = max(range(len(stages)), key=lambda i: stage_ms[i] if (stages[i][3] or stages[i][4]) else -1)
    dname, _, _, dfl, dby = stages[dom_i]
    dms = stage_ms[dom_i]
    if dfl:
        roof = {"kernel": dname, "bound": "tensor", "achieved": round(dfl / (dms * 1e-3) / 1e12, 1),
                "peak": round(fp8_peak, 1), "unit": "TFLOP/s"}
    else:
        roof = {"kernel": dname, "bound": "hbm", "achieved": round(dby / (dms * 1e-3) / 1e9, 1),
                "peak": round(hbm, 1), "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = traffic.get(dname)
    roof["peak_source"] = (f"{peak_src}: fp8 = 2 x bf16 burst {bf16_tf} TF/s" if dfl else f"{peak_src}: HBM copy {hbm} GB/s")

    # block-scaled forward at the same shapes (1x128 x tiles, 128x128 W blocks), timed alone
    blk = run_block_scaled(g, torch, x, wm, stream, flush, args.steps)
    # end to end through the public API with host buffers
    e2e = run_e2e(g, torch, x_h, w_h, dy_h, stream, args.steps, step_flops)

    launches = sum(s[2] for s in stages) * args.steps
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/e5m2 x fp32-accumulate -> bf16", "data": "synthetic",
        "config": {"workload": "gpt2s_upproj_train_step", "M_tokens": M, "d_model": K, "d_ff": N,
                   "step": "(requantise W || quantise x), fwd GEMM, quantise dy, dgrad + wgrad in one grouped launch, 3 history commits; one CUDA graph on two streams",
                   "scaling": "per-tensor delayed, amax history 16", "global_batch_tokens": M * world,
                   "l2": "256 MiB buffer written between timed steps (flush)", "parallelism": f"dp{world} (independent batches)"},
        "roofline": roof,
        "kernels": kernels,
        "kernels_note": "per-stage CUDA-event times of the same stages launched eagerly in the timed loop, each "
                        "behind an L2 flush (cold L2; sum %.4f ms vs the graph step)" % probe_step_ms,
        "block_scaled_fwd": blk,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed": round(wall, 4),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_full_step()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def run_block_scaled(g, torch, x, wm, stream, flush, steps):
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device="cuda")
    xq, wq, wqT = u8(M, K), u8(K, N), u8(N, K)
    xsi = torch.empty(M, K // 128, dtype=torch.float32, device="cuda")
    wsi = torch.empty(K // 128, N // 128, dtype=torch.float32, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    B = g.FP8_GRAN_BLOCK_128x128
    calls = [
        ("requant_w_block", lambda: g.fp8_requantize_weights(wm, K, N, B, 0, None, wq, wqT, wsi), 0.0, K * N * 4.0),
        ("quant_x_1x128", lambda: g.fp8_quantize(x, M, K, K, 0, g.FP8_GRAN_TILE_1x128, 0, None, xq, None, xsi),
         0.0, M * K * 3.0 + M * K / 128 * 4),
        ("gemm_fwd_block_scaled", lambda: g.fp8_scaled_mm(xq, 0, wqT, 0, M, N, K, K, K, B, xsi, wsi, y, N),
         2.0 * M * N * K, 0.0),
    ]
    with torch.cuda.stream(stream):
        for _, fn, _, _ in calls:
            fn()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(steps)]
        for k in range(steps):
            flush.zero_()
            ev[k][0].record(stream)
            for i, (_, fn, _, _) in enumerate(calls):
                fn()
                ev[k][i + 1].record(stream)
        torch.cuda.synchronize()
    out = {}
    hbm, bf16_tf, _ = load_peaks()
    for i, (name, _, fl, by) in enumerate(calls):
        ms = sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(steps)) / steps
        d = {"ms": round(ms, 5)}
        if fl:
            d.update(achieved=round(fl / (ms * 1e-3) / 1e12, 1), unit="TFLOP/s", frac=round(fl / (ms * 1e-3) / 1e12 / (2 * bf16_tf), 4))
        else:
            d.update(achieved=round(by / (ms * 1e-3) / 1e9, 1), unit="GB/s", frac=round(by / (ms * 1e-3) / 1e9 / hbm, 4))
        out[name] = d
    return out


def run_e2e(g, torch, x_h, w_h, dy_h, stream, steps, step_flops):
    """The same step through the public API (requantise + linear forward + linear backward
    + commits) with host inputs: pinned host -> device copies of x, W and dy and device ->
    host copies of y, dx and dW inside the timed region, every step. Steps alternate between
    two sets of device inputs and outputs (and host result buffers), so one step's uploads
    and compute overlap the previous step's downloads."""
    import numpy as np
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    xh, wh, dyh = pin(x_h), pin(w_h), pin(dy_h)
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device="cuda")
    sets = []
    for _ in range(2):
        sets.append(dict(x=bf(M, K), wm=bf(K, N), dy=bf(M, N), y=bf(M, N), dx=bf(M, K), dw=bf(K, N),
                         yh=torch.empty(M, N, dtype=torch.bfloat16).pin_memory(),
                         dxh=torch.empty(M, K, dtype=torch.bfloat16).pin_memory(),
                         dwh=torch.empty(K, N, dtype=torch.bfloat16).pin_memory(),
                         ev_xw=torch.cuda.Event(), ev_dy=torch.cuda.Event(), ev_fwd=torch.cuda.Event(),
                         ev_done=torch.cuda.Event(), ev_out=torch.cuda.Event(), used=False))
    wq, wqT, xq, xqT, dyq, dyqT = u8(K, N), u8(N, K), u8(M, K), u8(K, M), u8(M, N), u8(N, M)
    wst, xst, gst = g.TensorState(HIST), g.TensorState(HIST), g.TensorState(HIST)
    D, T = g.FP8_SCALE_DELAYED, g.FP8_GRAN_TENSOR
    wsb = g.fp8_linear_bwd_workspace_bytes(M, K, N)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    count = [0]

    def one():
        b = sets[count[0] % 2]
        count[0] += 1
        if b["used"]:
            s_in.wait_event(b["ev_done"])  # this set's previous step has read its inputs
            stream.wait_event(b["ev_out"])  # ... and its outputs are on the host
        b["used"] = True
        with torch.cuda.stream(s_in):
            b["x"].copy_(xh, non_blocking=True)
            b["wm"].copy_(wh, non_blocking=True)
            b["ev_xw"].record(s_in)
            b["dy"].copy_(dyh, non_blocking=True)
            b["ev_dy"].record(s_in)
        stream.wait_event(b["ev_xw"])
        g.fp8_requantize_weights(b["wm"], K, N, T, D, wst, wq, wqT)
        g.fp8_linear_fwd(b["x"], M, K, N, wqT, wst, None, xst, T, D, xq, xqT, None, b["y"])
        b["ev_fwd"].record(stream)
        stream.wait_event(b["ev_dy"])
        g.fp8_linear_bwd_ws(b["dy"], M, K, N, xqT, xst, wq, wst, gst, D, dyq, dyqT, b["dx"], b["dw"], ws, wsb)
        g.fp8_history_commit_many([wst, xst, gst])
        b["ev_done"].record(stream)
        s_out.wait_event(b["ev_fwd"])
        with torch.cuda.stream(s_out):
            b["yh"].copy_(b["y"], non_blocking=True)
        s_out.wait_event(b["ev_done"])
        with torch.cuda.stream(s_out):
            b["dxh"].copy_(b["dx"], non_blocking=True)
            b["dwh"].copy_(b["dw"], non_blocking=True)
            b["ev_out"].record(s_out)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for _ in range(steps):
            one()
        stream.wait_stream(s_out)  # the last step's results are on the host
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(step_flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(2 * (M * K + K * N + M * N)),
            "d2h_bytes_per_step": int(2 * (M * N + M * K + K * N))}


# --------------------------------------------------------------------------------------
# per-kernel sweep over the five workloads' shapes (not part of the bench line)
# --------------------------------------------------------------------------------------
# name, M, N, K, format of A, format of B, block scaled
SWEEP_GEMMS = [
    ("tiny_fwd", 256, 512, 128, 0, 0, False),
    ("gpt2s_fwd", 8192, 3072, 768, 0, 0, False),
    ("gpt2s_dgrad", 8192, 768, 3072, 1, 0, False),
    ("gpt2s_wgrad", 768, 3072, 8192, 0, 1, False),
    ("bwd_dgrad", 16384, 1024, 4096, 1, 0, False),
    ("bwd_wgrad", 1024, 4096, 16384, 0, 1, False),
    ("fine_fwd_block", 16384, 14336, 4096, 0, 0, True),
    ("fine_fwd_tensor", 16384, 14336, 4096, 0, 0, False),
    ("loop_fwd", 32768, 6144, 1536, 0, 0, False),
    ("loop_dgrad", 32768, 1536, 6144, 1, 0, False),
    ("loop_wgrad", 1536, 6144, 32768, 0, 1, False),
    # the same kernels on the other projections of a GPT-2-small block (8192 tokens, d 768)
    ("gpt2s_qkv_fwd", 8192, 2304, 768, 0, 0, False),
    ("gpt2s_down_fwd", 8192, 768, 3072, 0, 0, False),
    ("gpt2s_attn_out_fwd", 8192, 768, 768, 0, 0, False),
]
# name, rows, cols, format, granularity (0 tensor, 1 1x128, 2 128x128), transposed copy
SWEEP_CASTS = [
    ("gpt2s_dy_e5m2", 8192, 3072, 1, 0, True),
    ("bwd_dy_e5m2", 16384, 4096, 1, 0, True),
    ("bwd_x_e4m3", 16384, 1024, 0, 0, True),
    ("bwd_dy_e5m2_rowmajor", 16384, 4096, 1, 0, False),
    ("fine_x_1x128", 16384, 4096, 0, 1, False),
    ("fine_w_128x128", 4096, 14336, 0, 2, True),
    ("loop_dy_e5m2", 32768, 6144, 1, 0, True),
]
# the fused and multi-tensor entry points at the delayed-loop shapes (delayed scaling with one
# history entry): the optimizer-step update fused with W's refresh, W's and x's casts in one
# launch, and the forward GEMM that also writes the FP8 codes of its output
SWEEP_FUSED = ["loop_w_update", "loop_x_w_many", "loop_fwd_quant_out"]


def run_sweep(args):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import fp8_mixed_precision_saturating_gb300 as g
    torch.cuda.set_device(0)
    hbm, bf16_tf, _ = load_peaks()
    fp8_peak = 2 * bf16_tf
    gen = torch.Generator(device="cuda").manual_seed(0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    only = set(args.only.split(",")) if args.only else None

    def codes(rows, cols, fmt):
        # finite codes of either sign: magnitudes below the NaN / inf encodings
        mag = torch.randint(0, 0x70, (rows, cols), generator=gen, device="cuda", dtype=torch.int32)
        sgn = torch.randint(0, 2, (rows, cols), generator=gen, device="cuda", dtype=torch.int32) << 7
        return (mag | sgn).to(torch.uint8)

    def timed(fn, iters):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(iters):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    for name, m, n, k, fa, fb, blk in SWEEP_GEMMS:
        if only and name not in only:
            continue
        A, B = codes(m, k, fa), codes(n, k, fb)
        C = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        if blk:
            sa = torch.rand(m, k // 128, generator=gen, device="cuda") * 1e-2
            sb = torch.rand(k // 128, n // 128, generator=gen, device="cuda") * 1e-2
            gran = g.FP8_GRAN_BLOCK_128x128
        else:
            sa = torch.full((1,), 1e-2, device="cuda")
            sb = torch.full((1,), 1e-2, device="cuda")
            gran = g.FP8_GRAN_TENSOR
        # per-tensor GEMMs through the workspace entry point (split K where the shape asks)
        wsb = 0 if blk else g.fp8_scaled_mm_workspace_bytes(m, n, k)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
        if blk:
            fn = lambda: g.fp8_scaled_mm(A, fa, B, fb, m, n, k, k, k, gran, sa, sb, C, n)
        else:
            fn = lambda: g.fp8_scaled_mm_ws(A, fa, B, fb, m, n, k, k, k, gran, sa, sb, C, n, ws, wsb)
        ms = timed(fn, args.steps)
        tf = 2.0 * m * n * k / (ms * 1e-3) / 1e12
        out = {"sweep": "gemm", "name": name, "M": m, "N": n, "K": k, "block_scaled": blk,
               "split_k_workspace": wsb, "ms": round(ms, 5), "TFLOP/s": round(tf, 1),
               "frac_fp8_peak": round(tf / fp8_peak, 4)}
        if not blk:  # context: the vendor library's FP8 GEMM (the pages' torch._scaled_mm) on the same shape
            out["torch_scaled_mm"] = library_scaled_mm(torch, timed, A, fa, B, fb, m, n, k)
        print(json.dumps(out))
        del A, B, C
    for name, r, c, fmt, gran, tr in SWEEP_CASTS:
        if only and name not in only:
            continue
        x = torch.randn(r, c, generator=gen, device="cuda").to(torch.bfloat16)
        q = torch.empty(r, c, dtype=torch.uint8, device="cuda")
        qT = torch.empty(c, r, dtype=torch.uint8, device="cuda") if tr else None
        st = g.TensorState()
        if gran == 0:
            fn = lambda: g.fp8_quantize(x, r, c, c, fmt, 0, g.FP8_SCALE_CURRENT, st, q, qT)
            by = r * c * (3.0 + (1 if tr else 0))
        elif gran == 1:
            si = torch.empty(r, c // 128, device="cuda")
            fn = lambda: g.fp8_quantize(x, r, c, c, fmt, 1, 0, None, q, None, si)
            by = r * c * 3.0 + r * c / 128 * 4
        else:
            si = torch.empty(r // 128, c // 128, device="cuda")
            fn = lambda: g.fp8_quantize(x, r, c, c, fmt, 2, 0, None, q, qT, si)
            by = r * c * (3.0 + (1 if tr else 0)) + r * c / 16384 * 4
        ms = timed(fn, args.steps)
        gbs = by / (ms * 1e-3) / 1e9
        out = {"sweep": "cast", "name": name, "rows": r, "cols": c, "ms": round(ms, 5),
               "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)}
        if gran == 0:  # the current-scaling amax pass re-reads x: not algorithmic, reported apart
            st2 = g.TensorState(2)
            st2.amax_history[0] = st.amax_cur[0]  # the tensor's own amax: no saturation
            st2.hist_count[0] = 1
            ms_c = timed(lambda: g.fp8_quantize(x, r, c, c, fmt, 0, g.FP8_SCALE_DELAYED, st2, q, qT), args.steps)
            out.update(ms_cast_only=round(ms_c, 5), cast_only_GB_s=round(by / (ms_c * 1e-3) / 1e9, 1))
        print(json.dumps(out))
        del x, q, qT
    for name in SWEEP_FUSED:
        if only and name not in only:
            continue
        print(json.dumps(sweep_fused(g, torch, name, timed, codes, hbm, fp8_peak, args.steps)))
    if only is None or "delayed_loop" in only:
        run_delayed_loop(g, torch, fp8_peak)
    g.fp8_poll_device_error()


def library_scaled_mm(torch, timed, A, fa, B, fb, m, n, k):
    """torch._scaled_mm (cuBLASLt) on the same codes, per-tensor unit scales, bf16 output,
    timed like the sweep's own GEMMs; a comparison figure, not part of the library."""
    dt = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}
    try:
        a, b = A.view(dt[fa]), B.view(dt[fb])
        one = torch.ones((), device="cuda")
        ms = timed(lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16), 15)
        return {"ms": round(ms, 5), "TFLOP/s": round(2.0 * m * n * k / (ms * 1e-3) / 1e12, 1)}
    except Exception as e:  # a format pair or shape the library does not take
        return {"unavailable": str(e).splitlines()[0][:120]}


def sweep_fused(g, torch, name, timed, codes, hbm, fp8_peak, steps):
    """One SWEEP_FUSED entry: its states get one history entry from an untimed first call
    (the bootstrap) and a commit; the timed calls then cast with the history's scale."""
    D = g.FP8_SCALE_DELAYED
    gen = torch.Generator(device="cuda").manual_seed(7)
    u8 = lambda *sh: torch.empty(*sh, dtype=torch.uint8, device="cuda")
    tokens, d = 32768, 1536
    n = 4 * d
    if name == "loop_w_update":
        w = (torch.randn(d, n, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
        delta = torch.randn(d, n, generator=gen, device="cuda") * 1e-3
        st, wq, wqT = g.TensorState(), u8(d, n), u8(n, d)
        fn = lambda: g.fp8_update_requantize_weights(w, delta, d, n, D, st, wq, wqT)
        states, by, fl = [st], d * n * 10.0, 0.0  # W 2 + delta 4 read, W' 2 + codes 2 written
    elif name == "loop_x_w_many":
        x = torch.randn(tokens, d, generator=gen, device="cuda").to(torch.bfloat16)
        w = (torch.randn(d, n, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
        sx, sw = g.TensorState(), g.TensorState()
        outs = [u8(tokens, d), u8(d, tokens), u8(d, n), u8(n, d)]  # (held for the jobs' lifetime)
        jobs = [g.quant_job(x, tokens, d, d, g.FP8_E4M3, D, sx, outs[0], outs[1]),
                g.quant_job(w, d, n, n, g.FP8_E4M3, D, sw, outs[2], outs[3])]
        fn = lambda: g.fp8_quantize_many(jobs)
        states, by, fl = [sx, sw], (tokens * d + d * n) * 4.0, 0.0
    else:
        A, B = codes(tokens, d, 0), codes(n, d, 0)
        sa, sb = torch.full((1,), 1e-2, device="cuda"), torch.full((1,), 1e-2, device="cuda")
        C, Cq, sc = torch.empty(tokens, n, dtype=torch.bfloat16, device="cuda"), u8(tokens, n), g.TensorState()
        fn = lambda: g.fp8_scaled_mm_quant(A, 0, B, 0, tokens, n, d, d, d, sa, sb, C, n, g.FP8_E4M3, sc, Cq)
        states, by, fl = [sc], 0.0, 2.0 * tokens * n * d
    fn()
    g.fp8_history_commit_many(states)
    ms = timed(fn, steps)
    out = {"sweep": "fused", "name": name, "ms": round(ms, 5)}
    if fl:
        tf = fl / (ms * 1e-3) / 1e12
        out.update({"TFLOP/s": round(tf, 1), "frac_fp8_peak": round(tf / fp8_peak, 4)})
    else:
        gbs = by / (ms * 1e-3) / 1e9
        out.update({"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)})
    return out


def run_delayed_loop(g, torch, fp8_peak, layers=12, steps=50, tokens=32768, d=1536, hist=16):
    """The delayed-scaling training loop at full size through the public API: every step and
    layer refreshes W with its optimizer step and re-quantises it (one fused pass), casts x
    and dy with the delayed scales, runs the forward, dgrad and wgrad GEMMs and commits the
    three amaxes. x, dy and the per-layer steps are drawn once (synthetic, seeded); the timed
    region is the whole trajectory after one untimed step."""
    n = 4 * d
    gen = torch.Generator(device="cuda").manual_seed(5)
    x = (torch.randn(tokens, d, generator=gen, device="cuda")).to(torch.bfloat16)
    dy = (torch.randn(tokens, n, generator=gen, device="cuda") * 1e-3).to(torch.bfloat16)
    u8 = lambda *sh: torch.empty(*sh, dtype=torch.uint8, device="cuda")
    bf = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device="cuda")
    W = [(torch.randn(d, n, generator=gen, device="cuda") * 0.02).to(torch.bfloat16) for _ in range(layers)]
    delta = [torch.randn(d, n, generator=gen, device="cuda") * 1e-3 for _ in range(layers)]
    st = [[g.TensorState(hist) for _ in range(3)] for _ in range(layers)]
    wq, wqT = [u8(d, n) for _ in range(layers)], [u8(n, d) for _ in range(layers)]
    xq, xqT, dyq, dyqT = u8(tokens, d), u8(d, tokens), u8(tokens, n), u8(n, tokens)
    y, dx, dw = bf(tokens, n), bf(tokens, d), bf(d, n)
    wsb = g.fp8_linear_bwd_workspace_bytes(tokens, d, n)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    D, T = g.FP8_SCALE_DELAYED, g.FP8_GRAN_TENSOR

    def layer_step(l):  # the layer API: 6 launches (update + requantise, x cast, forward GEMM,
        ws_, xs, gs = st[l]  # dy cast, grouped dgrad + wgrad, history commit)
        g.fp8_update_requantize_weights(W[l], delta[l], d, n, D, ws_, wq[l], wqT[l])
        g.fp8_linear_fwd(x, tokens, d, n, wqT[l], ws_, None, xs, T, D, xq, xqT, None, y)
        g.fp8_linear_bwd_ws(dy, tokens, d, n, xqT, xs, wq[l], ws_, gs, D, dyq, dyqT, dx, dw, ws, wsb)
        g.fp8_history_commit_many([ws_, xs, gs])

    for l in range(layers):  # untimed first step (bootstrap casts)
        layer_step(l)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps - 1):
        for l in range(layers):
            layer_step(l)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    flops = 3 * 2.0 * tokens * d * n * layers * (steps - 1)
    tf = flops / (ms * 1e-3) / 1e12
    ov = sum(int(s.counters[0]) for lay in st for s in lay)
    print(json.dumps({"sweep": "delayed_loop", "layers": layers, "steps_timed": steps - 1, "tokens": tokens, "d": d,
                      "ms_total": round(ms, 3), "ms_per_layer_step": round(ms / (layers * (steps - 1)), 4),
                      "TFLOP/s": round(tf, 1), "frac_fp8_peak": round(tf / fp8_peak, 4),
                      "launches_per_layer_step": 6, "overflow_counts_total": ov}))


# --------------------------------------------------------------------------------------
# CPU oracle arm
# --------------------------------------------------------------------------------------
def oracle_step(tokens: int):
    """One oracle pass of the step's arithmetic on `tokens` of the M tokens (W in full).
    Returns the GEMM FLOPs it covered."""
    from datagen import workload_inputs, lognormal_grad_bf16
    from oracle import fp8, gemm, quant
    w = oracle_step.cache if hasattr(oracle_step, "cache") else None
    if w is None:
        w = workload_inputs("gpt2s_upproj_fwd")
        w["dy"] = lognormal_grad_bf16(2002, (M, N))
        oracle_step.cache = w
    x, dy = w["x"][:tokens], w["dy"][:tokens]
    ow = quant.quantize_tensor(w["w"], fp8.E4M3)
    ox = quant.quantize_tensor(x, fp8.E4M3)
    og = quant.quantize_tensor(dy, fp8.E5M2)
    gemm.scaled_mm(ox["q"], fp8.E4M3, ow["qT"], fp8.E4M3, ox["d"], ow["d"])
    gemm.scaled_mm(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"])
    gemm.scaled_mm(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"])
    return 3 * 2.0 * tokens * N * K


def cpu_baseline_full_step(steps: int = 3):
    oracle_step(64)  # load inputs
    t0 = time.perf_counter()
    fl = sum(oracle_step(M) for _ in range(steps))
    dt = time.perf_counter() - t0
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{steps} full steps ({M} tokens each): numpy oracle casts (one thread) and fp64 BLAS "
                      f"matmuls (all cores); {dt:.1f} s"}


def run_reference(args):
    rank, _, world = env_rank()
    if rank != 0:
        return
    tokens = 2048
    for _ in range(args.warmup):
        oracle_step(tokens)
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += oracle_step(tokens)
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    sample = f"{tokens} of {M} tokens per step (W in full), numpy oracle, fp64 BLAS matmuls"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": "gpt2s_upproj_train_step", "M_tokens": M, "d_model": K, "d_ff": N},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="time every workload's GEMM and cast shapes instead")
    ap.add_argument("--only", default="", help="comma-separated sweep entries")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
