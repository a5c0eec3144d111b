#!/usr/bin/env python
"""Benchmark of the FP8 up-projection hot path on GB300.

Headline (the JSON line's value): the fine-grained-scaling forward at its full size.
  x bf16 [16384 x 4096] = z * std_c (z ~ N(0,1), std_c = 10^U(-1,1) per channel),
  W bf16 [4096 x 14336] ~ N(0, 0.02). One step is one pass of the hot path:
    W's E4M3 cast with one scale per 128 x 128 block into W_q^T [14336 x 4096] (the weight
      cache refresh)                                         || on a second stream
    x's E4M3 cast with one scale per 1 x 128 row tile into x_q [16384 x 4096]
    the block-scaled GEMM y = bf16( sum_kb d_x[i,kb] d_w[kb,j/128] P_ij,kb ) [16384 x 14336]
  value = the GEMM's 2MNK over the step time; the roofline is the block-scaled GEMM's.
The step is captured into a CUDA graph; each timed step replays it between CUDA events after
writing a 256 MiB buffer (the L2 flush, not timed). Per-kernel times come from the same stages
launched eagerly in the same loop, each behind a flush.

Sub-records in the same line, each with its own roofline, kernel times and oracle CPU baseline:
  finegrained_upproj_fwd_mx  the headline's shapes and inputs with MX scales (a power-of-two
                    UE8M0 scale per 32 contraction elements, applied by the tensor cores):
                    W's cast down its columns (written as W_q^T) || x's cast along its rows,
                    the block-scaled (kind::mxf8f6f4) GEMM
  backward_upproj   M=16384, K=1024, N=4096: dy's E5M2 cast (current scaling, dy_q only),
                    dgrad and wgrad in one grouped launch, the wgrad reading x_q and dy_q
                    MN-major (no transposed copies)
  delayed_loop      32768 tokens, d 1536 -> 6144, history 16: one layer-step (optimizer step
                    fused with W's refresh, x cast, forward, dy cast, dgrad + wgrad, commit)
                    and the 12-layer step
  gpt2s_train_step  8192 tokens, d 768 -> 3072: the whole training step with delayed scaling

--impl reference times the CPU oracle (test infrastructure) on a bounded sample of the
headline's step on the host cores.
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
# the fine-grained forward (headline), the backward, the delayed loop and GPT-2 small
FINE = dict(M=16384, K=4096, N=14336)
BWD = dict(M=16384, K=1024, N=4096)
LOOP = dict(M=32768, K=1536, N=6144, layers=12, hist=16)
GPT2 = dict(M=8192, K=768, N=3072, hist=16)
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
# per-launch DRAM counters (profiles/traffic_per_launch.txt)
# --------------------------------------------------------------------------------------
# The sources that decide each stage's kernel and launch (kernel body, its headers, the
# host code that picks and launches it): a stage's DRAM counters stay valid while these hash
# the same as when the counters were taken.
_CAST_SOURCES = ("quant.cu", "cast.cuh", "ptx.cuh", "kernels.h", "api.cu")
_GEMM_SOURCES = ("gemm.cu", "cast.cuh", "ptx.cuh", "kernels.h", "api.cu")
STAGE_SOURCES = {
    # GPT-2-small training step
    "requant_w": _CAST_SOURCES, "quant_x": _CAST_SOURCES, "quant_dy": _CAST_SOURCES,
    "gemm_fwd": _GEMM_SOURCES, "gemm_bwd": _GEMM_SOURCES,
    # fine-grained forward (headline), and the same shapes with MX scales
    "fine_cast_w": _CAST_SOURCES, "fine_cast_x": _CAST_SOURCES, "fine_gemm": _GEMM_SOURCES,
    "mx_cast_w": _CAST_SOURCES, "mx_cast_x": _CAST_SOURCES, "mx_gemm": _GEMM_SOURCES,
    # backward
    "bwd_cast_dy": _CAST_SOURCES, "bwd_gemm": _GEMM_SOURCES,
    # delayed loop, one layer-step
    "loop_update_w": _CAST_SOURCES, "loop_cast_x": _CAST_SOURCES, "loop_gemm_fwd": _GEMM_SOURCES,
    "loop_cast_dy": _CAST_SOURCES, "loop_gemm_bwd": _GEMM_SOURCES,
}


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
    """Seed offset of rank r's own batch: rank 0 uses the workloads' own seeds."""
    return (0, 0) if rank == 0 else (10 * rank, 10 * rank + 1)


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


# --------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------
class Stage:
    """One launch of a step: name (a STAGE_SOURCES key), the call, the kernels it launches and
    its algorithmic work (GEMM FLOPs, or bytes a cast must move)."""

    def __init__(self, name, fn, launches, flops=0.0, nbytes=0.0):
        self.name, self.fn, self.launches, self.flops, self.nbytes = name, fn, launches, flops, nbytes


def time_step(torch, stream, flush, enqueue_step, stages, steps, warmup, before_replays=None, clocks=None):
    """Capture enqueue_step() (the whole step, possibly on several streams) into one CUDA graph
    on `stream`, then run warmup + steps iterations. An iteration: flush L2 (untimed), replay
    the graph between two events on `stream`; then launch every stage eagerly, each behind its
    own flush and between its own events (cold L2, per-kernel times). Returns per-step graph
    times (ms), per-stage mean times (ms) and the wall time of the timed iterations."""
    with torch.cuda.stream(stream):
        for st in stages:  # eager pass: kernel attributes, plans and caches
            st.fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            enqueue_step()
        if before_replays is not None:
            before_replays()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in stages]

        def one():
            flush.zero_()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            for (a, b), st in zip(ev, stages):
                flush.zero_()
                a.record(stream)
                st.fn()
                b.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1), [a.elapsed_time(b) for a, b in ev]

        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.start()
            time.sleep(0.3)  # let the sampler see the first samples
        wall0 = time.perf_counter()
        res = [one() for _ in range(steps)]
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    step_ms = [t for t, _ in res]
    stage_ms = [sum(r[1][i] for r in res) / steps for i in range(len(stages))]
    return step_ms, stage_ms, wall


def kernel_records(stages, stage_ms, hbm, fp8_peak):
    out = {}
    for st, ms in zip(stages, stage_ms):
        kd = {"ms": round(ms, 5), "launches": st.launches}
        if st.flops:
            tf = st.flops / (ms * 1e-3) / 1e12
            kd.update(achieved=round(tf, 1), unit="TFLOP/s", frac=round(tf / fp8_peak, 4))
        elif st.nbytes:
            gbs = st.nbytes / (ms * 1e-3) / 1e9
            kd.update(achieved=round(gbs, 1), unit="GB/s", frac=round(gbs / hbm, 4))
        out[st.name] = kd
    return out


def roofline(stages, stage_ms, hbm, bf16_tf, peak_src, name=None):
    """The roofline object of one stage: the named one, else the one with algorithmic work that
    took longest. achieved = algorithmic work of one launch / its mean CUDA-event duration."""
    fp8_peak = 2.0 * bf16_tf
    idx = [i for i, st in enumerate(stages) if st.flops or st.nbytes]
    if name is not None:
        i = next(i for i in idx if stages[i].name == name)
    else:
        i = max(idx, key=lambda j: stage_ms[j])
    st, ms = stages[i], stage_ms[i]
    if st.flops:
        r = {"kernel": st.name, "bound": "tensor", "achieved": round(st.flops / (ms * 1e-3) / 1e12, 1),
             "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
             "peak_source": f"{peak_src}: fp8 = 2 x bf16 burst {bf16_tf} TF/s"}
    else:
        r = {"kernel": st.name, "bound": "hbm", "achieved": round(st.nbytes / (ms * 1e-3) / 1e9, 1),
             "peak": round(hbm, 1), "unit": "GB/s", "peak_source": f"{peak_src}: HBM copy {hbm} GB/s"}
    r["frac"] = round(r["achieved"] / r["peak"], 4)
    r["traffic"] = traffic_table().get(st.name)
    return r


def dev_bf16(torch, bits):
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def run_gpu(args):
    rank, local_rank, world = env_rank()
    # the oracle's CPU legs run first, in child processes, before this process touches the GPU
    cpu = cpu_baselines() if (rank == 0 and world == 1 and not args.no_cpu_baseline) else {}
    import torch

    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    import fp8_mixed_precision_saturating_gb300 as g

    hbm, bf16_tf, peak_src = load_peaks()
    fp8_peak = 2.0 * bf16_tf
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    ctx = dict(torch=torch, g=g, stream=stream, flush=flush, hbm=hbm, bf16_tf=bf16_tf, peak_src=peak_src,
               fp8_peak=fp8_peak, rank=rank, world=world)

    # ---- headline: the fine-grained forward at full size
    clocks = Clocks(local_rank)
    if world > 1:
        torch.distributed.barrier()
    head = bench_finegrained(ctx, args.steps, args.warmup, clocks)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(head["step_ms"]), world, "cuda")
    value = weak_scaling_value(head["step_flops"], args.steps, world, total_ms)

    # ---- sub-records (rank 0 reports them; every rank runs the same work)
    subs = {}
    if not args.headline_only:
        want = set(args.records.split(",")) if args.records else None
        runs = [("finegrained_upproj_fwd_mx", lambda: bench_finegrained_mx(ctx, args.steps, args.warmup)),
                ("backward_upproj", lambda: bench_backward(ctx, max(5, args.steps // 2), args.warmup)),
                ("delayed_loop", lambda: bench_delayed_loop(ctx, max(3, args.steps // 4), args.warmup)),
                ("gpt2s_train_step", lambda: bench_gpt2(ctx, args.steps, args.warmup))]
        for name, run in runs:
            if want is None or name in want:
                subs[name] = run()
        for k, v in subs.items():
            if k in cpu:
                v["cpu_baseline"] = cpu[k]
    g.fp8_poll_device_error()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3, fp32 accumulate and fp32 block scales -> bf16",
        "data": "synthetic",
        "config": {"workload": "finegrained_upproj_fwd", "M_tokens": FINE["M"], "d_model": FINE["K"],
                   "d_ff": FINE["N"],
                   "x": "bf16 z * 10^U(-1,1) per channel; E4M3 with one fp32 scale per 1x128 row tile",
                   "W": "bf16 N(0, 0.02); E4M3 with one fp32 scale per 128x128 block, cached as W_q^T",
                   "step": "(W block cast || x tile cast on two streams), block-scaled GEMM; one CUDA graph",
                   "global_batch_tokens": FINE["M"] * world,
                   "l2": "256 MiB buffer written before every timed step and stage (flush); inputs 134 + 117 MB",
                   "parallelism": f"dp{world} (independent batches)"},
        "roofline": head["roofline"],
        "kernels": head["kernels"],
        "kernels_note": "per-stage CUDA-event times of the same stages launched eagerly in the timed loop, each "
                        "behind an L2 flush (cold L2)",
        "e2e": head["e2e"],
        "gpu_launches": head["launches"],
        "clocks": clk,
        "wall_s_timed": round(head["wall"], 4),
    }
    line.update(subs)
    if "finegrained" in cpu:
        line["cpu_baseline"] = cpu["finegrained"]
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_finegrained(ctx, steps, warmup, clocks):
    """The headline step; its e2e leg through the public API with host buffers."""
    import numpy as np
    from datagen import workload_inputs, channel_scaled_bf16
    torch, g, stream, flush = ctx["torch"], ctx["g"], ctx["stream"], ctx["flush"]
    M, K, N = FINE["M"], FINE["K"], FINE["N"]
    w_in = workload_inputs("finegrained_fwd")
    x_h = w_in["x"] if ctx["rank"] == 0 else channel_scaled_bf16(4000 + rank_seeds(ctx["rank"])[0], (M, K))
    w_h = w_in["w"]
    x, wm = dev_bf16(torch, x_h), dev_bf16(torch, w_h)
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device="cuda")
    xq, wqT = u8(M, K), u8(N, K)
    xsi = torch.empty(M, K // 128, dtype=torch.float32, device="cuda")
    wsi = torch.empty(K // 128, N // 128, dtype=torch.float32, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    B, TL, CUR = g.FP8_GRAN_BLOCK_128x128, g.FP8_GRAN_TILE_1x128, g.FP8_SCALE_CURRENT
    flops = 2.0 * M * N * K
    stages = [
        Stage("fine_cast_w", lambda: g.fp8_requantize_weights(wm, K, N, B, CUR, None, None, wqT, wsi), 1,
              nbytes=K * N * 3.0 + (K // 128) * (N // 128) * 4),
        Stage("fine_cast_x", lambda: g.fp8_quantize(x, M, K, K, g.FP8_E4M3, TL, CUR, None, xq, None, xsi), 1,
              nbytes=M * K * 3.0 + M * (K // 128) * 4),
        Stage("fine_gemm", lambda: g.fp8_scaled_mm(xq, 0, wqT, 0, M, N, K, K, K, B, xsi, wsi, y, N), 1, flops=flops),
    ]
    side = torch.cuda.Stream()

    def enqueue():
        side.wait_stream(stream)
        stages[0].fn()
        with torch.cuda.stream(side):
            stages[1].fn()
        stream.wait_stream(side)
        stages[2].fn()

    step_ms, stage_ms, wall = time_step(torch, stream, flush, enqueue, stages, steps, warmup, clocks=clocks)
    e2e = e2e_finegrained(ctx, x_h, w_h, steps, flops)
    return {"step_ms": step_ms, "step_flops": flops, "wall": wall,
            "kernels": kernel_records(stages, stage_ms, ctx["hbm"], ctx["fp8_peak"]),
            "roofline": roofline(stages, stage_ms, ctx["hbm"], ctx["bf16_tf"], ctx["peak_src"], name="fine_gemm"),
            "e2e": e2e, "launches": 2 * len(stages) * steps}


def e2e_finegrained(ctx, x_h, w_h, steps, step_flops):
    """The headline step through the public API (fp8_requantize_weights + fp8_linear_fwd with
    block scaling) from pinned host buffers: x and W copied up and y copied down every step,
    inside the timed region. Steps alternate between two sets of device buffers (and host
    result buffers), so one step's uploads and compute overlap the previous step's download."""
    import numpy as np
    torch, g, stream = ctx["torch"], ctx["g"], ctx["stream"]
    M, K, N = FINE["M"], FINE["K"], FINE["N"]
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    xh, wh = pin(x_h), pin(w_h)
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device="cuda")
    B, CUR = g.FP8_GRAN_BLOCK_128x128, g.FP8_SCALE_CURRENT
    sets = []
    for _ in range(2):
        sets.append(dict(x=bf(M, K), wm=bf(K, N), y=bf(M, N),
                         yh=torch.empty(M, N, dtype=torch.bfloat16).pin_memory(),
                         ev_in=torch.cuda.Event(), ev_done=torch.cuda.Event(), ev_out=torch.cuda.Event(), used=False))
    xq, wqT = u8(M, K), u8(N, K)
    xsi = torch.empty(M, K // 128, dtype=torch.float32, device="cuda")
    wsi = torch.empty(K // 128, N // 128, dtype=torch.float32, device="cuda")
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    count = [0]

    def one():
        b = sets[count[0] % 2]
        count[0] += 1
        if b["used"]:
            s_in.wait_event(b["ev_done"])  # this set's previous step has read its inputs
            stream.wait_event(b["ev_out"])  # ... and its output is on the host
        b["used"] = True
        with torch.cuda.stream(s_in):
            b["wm"].copy_(wh, non_blocking=True)
            b["x"].copy_(xh, non_blocking=True)
            b["ev_in"].record(s_in)
        stream.wait_event(b["ev_in"])
        g.fp8_requantize_weights(b["wm"], K, N, B, CUR, None, None, wqT, wsi)
        g.fp8_linear_fwd(b["x"], M, K, N, wqT, None, wsi, None, B, CUR, xq, None, xsi, b["y"])
        b["ev_done"].record(stream)
        s_out.wait_event(b["ev_done"])
        with torch.cuda.stream(s_out):
            b["yh"].copy_(b["y"], non_blocking=True)
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
        stream.wait_stream(s_out)  # the last step's result is on the host
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(step_flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(2 * (M * K + K * N)), "d2h_bytes_per_step": int(2 * M * N),
            "api": "fp8_requantize_weights + fp8_linear_fwd (block scaling), pinned host buffers"}


def bench_finegrained_mx(ctx, steps, warmup):
    """The headline's shapes and inputs with MX scales: W's cast in groups of 32 down its
    columns (W_q^T and its scale bytes) beside x's cast in groups of 32 along its rows, then
    the GEMM on the tensor cores' block scaling."""
    from datagen import workload_inputs
    torch, g, stream, flush = ctx["torch"], ctx["g"], ctx["stream"], ctx["flush"]
    M, K, N = FINE["M"], FINE["K"], FINE["N"]
    w_in = workload_inputs("finegrained_fwd")
    x, wm = dev_bf16(torch, w_in["x"]), dev_bf16(torch, w_in["w"])
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device="cuda")
    xq, wqT = u8(M, K), u8(N, K)
    xsf, wsf = u8(-(-M // 128) * (K // 128) * 512), u8(-(-N // 128) * (K // 128) * 512)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    X, CUR = g.FP8_GRAN_MX_1x32, g.FP8_SCALE_CURRENT
    flops = 2.0 * M * N * K
    stages = [
        Stage("mx_cast_w", lambda: g.fp8_requantize_weights(wm, K, N, X, CUR, None, None, wqT, wsf), 1,
              nbytes=K * N * 3.0 + wsf.numel()),
        Stage("mx_cast_x", lambda: g.fp8_quantize(x, M, K, K, g.FP8_E4M3, X, CUR, None, xq, None, xsf), 1,
              nbytes=M * K * 3.0 + xsf.numel()),
        Stage("mx_gemm", lambda: g.fp8_scaled_mm(xq, 0, wqT, 0, M, N, K, K, K, X, xsf, wsf, y, N), 1, flops=flops),
    ]
    side = torch.cuda.Stream()

    def enqueue():
        side.wait_stream(stream)
        stages[0].fn()
        with torch.cuda.stream(side):
            stages[1].fn()
        stream.wait_stream(side)
        stages[2].fn()

    step_ms, stage_ms, _ = time_step(torch, stream, flush, enqueue, stages, steps, warmup)
    ms = sum(step_ms) / steps
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
            "steps": steps,
            "config": {"workload": "finegrained_upproj_fwd_mx", "M_tokens": M, "d_model": K, "d_ff": N,
                       "scaling": "E4M3 with a UE8M0 power-of-two scale per 32 contraction elements (x along its "
                                  "rows, W down its columns), applied by block-scaled MMAs",
                       "step": "(W cast || x cast on two streams), MX GEMM; one CUDA graph"},
            "roofline": roofline(stages, stage_ms, ctx["hbm"], ctx["bf16_tf"], ctx["peak_src"], name="mx_gemm"),
            "kernels": kernel_records(stages, stage_ms, ctx["hbm"], ctx["fp8_peak"])}


def bench_backward(ctx, steps, warmup):
    """dy's per-tensor E5M2 cast (current scaling: amax pass, then dy_q in one pass) and the
    grouped dgrad + wgrad launch, with x's and W's saved codes cast once beforehand. The wgrad
    problem reads x_q [M, K] and dy_q [M, N] MN-major, so no cast writes a transposed copy."""
    from datagen import workload_inputs
    torch, g, stream, flush = ctx["torch"], ctx["g"], ctx["stream"], ctx["flush"]
    M, K, N = BWD["M"], BWD["K"], BWD["N"]
    w_in = workload_inputs("upproj_bwd")
    x, wm, dy = dev_bf16(torch, w_in["x"]), dev_bf16(torch, w_in["w"]), dev_bf16(torch, w_in["dy"])
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device="cuda")
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    T, CUR = g.FP8_GRAN_TENSOR, g.FP8_SCALE_CURRENT
    xst, wst, gst = g.TensorState(), g.TensorState(), g.TensorState()
    wq, wqT, xq, dyq = u8(K, N), u8(N, K), u8(M, K), u8(M, N)
    dx, dw = bf(M, K), bf(K, N)
    with torch.cuda.stream(stream):
        g.fp8_requantize_weights(wm, K, N, T, CUR, wst, wq, wqT)
        g.fp8_quantize(x, M, K, K, g.FP8_E4M3, T, CUR, xst, xq, None)
    bwd = [g.mm_problem(xq, 0, dyq, 1, K, N, M, K, N, xst.scale_inv, gst.scale_inv, dw, N, mn_major=1),
           g.mm_problem(dyq, 1, wq, 0, M, K, N, N, N, gst.scale_inv, wst.scale_inv, dx, K)]
    wsb = g.fp8_scaled_mm_grouped_workspace_bytes(bwd)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    flops = 2 * 2.0 * M * N * K
    stages = [
        Stage("bwd_cast_dy", lambda: g.fp8_quantize(dy, M, N, N, g.FP8_E5M2, T, CUR, gst, dyq, None), 1,
              nbytes=M * N * 3.0),
        Stage("bwd_gemm", lambda: g.fp8_scaled_mm_grouped(bwd, ws, wsb), 1, flops=flops),
    ]

    def enqueue():
        for st in stages:
            st.fn()

    step_ms, stage_ms, _ = time_step(torch, stream, flush, enqueue, stages, steps, warmup)
    ms = sum(step_ms) / steps
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
            "steps": steps, "config": {"workload": "upproj_bwd", "M_tokens": M, "d_model": K, "d_ff": N,
                                       "dy": "bf16 sign * 1e-4 * exp(2 z); E5M2 per tensor, current scaling",
                                       "step": "dy cast (dy_q), dgrad + wgrad in one grouped launch, "
                                               "wgrad reading x_q and dy_q MN-major"},
            "roofline": roofline(stages, stage_ms, ctx["hbm"], ctx["bf16_tf"], ctx["peak_src"], name="bwd_gemm"),
            "kernels": kernel_records(stages, stage_ms, ctx["hbm"], ctx["fp8_peak"])}


def bench_delayed_loop(ctx, steps, warmup):
    """One layer-step of the delayed-scaling loop at full size, and the step of all 12 layers,
    through the layer API: the optimizer step fused with W's refresh (delta drawn once per
    layer), x's cast and the forward GEMM, dy's cast and the grouped dgrad + wgrad, the
    history commit. x and dy are the loop's (drawn once, shared by all layers)."""
    from datagen import workload_inputs, normal_bf16, perturbation_f32
    import numpy as np
    torch, g, stream, flush = ctx["torch"], ctx["g"], ctx["stream"], ctx["flush"]
    M, K, N, L, H = LOOP["M"], LOOP["K"], LOOP["N"], LOOP["layers"], LOOP["hist"]
    w_in = workload_inputs("delayed_loop")
    x, dy = dev_bf16(torch, w_in["x"]), dev_bf16(torch, w_in["dy"])
    W = [dev_bf16(torch, w) for w in w_in["w"]]
    delta = [torch.from_numpy(perturbation_f32(w_in["perturb_seed"](l, 1), (K, N), 1e-3)).cuda() for l in range(L)]
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device="cuda")
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    D, T = g.FP8_SCALE_DELAYED, g.FP8_GRAN_TENSOR
    st = [[g.TensorState(H) for _ in range(3)] for _ in range(L)]
    wq, wqT = [u8(K, N) for _ in range(L)], [u8(N, K) for _ in range(L)]
    xq, dyq = u8(M, K), u8(M, N)
    y, dx, dw = bf(M, N), bf(M, K), bf(K, N)
    wsb = g.fp8_linear_bwd_workspace_bytes(M, K, N)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")

    def layer_step(l):  # 6 launches: update + requantise, x cast, forward GEMM, dy cast, grouped bwd, commit
        ws_, xs, gs = st[l]
        g.fp8_update_requantize_weights(W[l], delta[l], K, N, D, ws_, wq[l], wqT[l])
        g.fp8_linear_fwd(x, M, K, N, wqT[l], ws_, None, xs, T, D, xq, None, None, y)
        g.fp8_linear_bwd_mn(dy, M, K, N, xq, xs, wq[l], ws_, gs, D, dyq, dx, dw, ws, wsb)
        g.fp8_history_commit_many([ws_, xs, gs])

    with torch.cuda.stream(stream):
        for l in range(L):  # the bootstrap step (current amaxes), untimed
            layer_step(l)
        torch.cuda.synchronize()
    ws0, xs0, gs0 = st[0]
    bwd = [g.mm_problem(xq, 0, dyq, 1, K, N, M, K, N, xs0.scale_inv, gs0.scale_inv, dw, N, mn_major=1),
           g.mm_problem(dyq, 1, wq[0], 0, M, K, N, N, N, gs0.scale_inv, ws0.scale_inv, dx, K)]
    fl = 2.0 * M * N * K
    stages = [
        Stage("loop_update_w", lambda: g.fp8_update_requantize_weights(W[0], delta[0], K, N, D, ws0, wq[0], wqT[0]), 1,
              nbytes=K * N * 10.0),
        Stage("loop_cast_x", lambda: g.fp8_quantize(x, M, K, K, g.FP8_E4M3, T, D, xs0, xq, None), 1, nbytes=M * K * 3.0),
        Stage("loop_gemm_fwd", lambda: g.fp8_scaled_mm_ws(xq, 0, wqT[0], 0, M, N, K, K, K, T, xs0.scale_inv,
                                                            ws0.scale_inv, y, N, ws, wsb), 1, flops=fl),
        Stage("loop_cast_dy", lambda: g.fp8_quantize(dy, M, N, N, g.FP8_E5M2, T, D, gs0, dyq, None), 1,
              nbytes=M * N * 3.0),
        Stage("loop_gemm_bwd", lambda: g.fp8_scaled_mm_grouped(bwd, ws, wsb), 1, flops=2 * fl),
        Stage("loop_commit", lambda: g.fp8_history_commit_many([ws0, xs0, gs0]), 1),
    ]
    step_ms, stage_ms, _ = time_step(torch, stream, flush, lambda: layer_step(0), stages, steps, warmup)
    layer_ms = sum(step_ms) / steps
    # the 12-layer step: one graph of all layers' launches, replayed behind a flush
    with torch.cuda.stream(stream):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for l in range(L):
                layer_step(l)
        ts = []
        for _ in range(warmup + steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
    full_ms = sum(ts[warmup:]) / steps
    ov = sum(int(s.counters[0]) for lay in st for s in lay)
    return {"value": round(3 * fl / (layer_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_layer_step": round(layer_ms, 5), "ms_per_12_layer_step": round(full_ms, 4),
            "value_12_layer_step": round(L * 3 * fl / (full_ms * 1e-3) / 1e12, 2), "steps": steps,
            "launches_per_layer_step": 6,
            "config": {"workload": "delayed_loop", "M_tokens": M, "d_model": K, "d_ff": N, "layers": L,
                       "scaling": "per-tensor delayed, amax history 16 (after one untimed bootstrap step)",
                       "delta": "optimizer step N(0, 1e-3) per element, drawn once per layer"},
            "overflow_counts_total": ov,
            "roofline": roofline(stages, stage_ms, ctx["hbm"], ctx["bf16_tf"], ctx["peak_src"]),
            "kernels": kernel_records(stages, stage_ms, ctx["hbm"], ctx["fp8_peak"])}


def bench_gpt2(ctx, steps, warmup):
    """The GPT-2-small-shaped training step with delayed scaling: (W's refresh || x's cast on
    two streams), the forward GEMM, dy's cast, dgrad + wgrad in one grouped launch, the three
    history commits; the states start empty, so the first replay is the bootstrap step."""
    from datagen import workload_inputs, lognormal_grad_bf16
    torch, g, stream, flush = ctx["torch"], ctx["g"], ctx["stream"], ctx["flush"]
    M, K, N, H = GPT2["M"], GPT2["K"], GPT2["N"], GPT2["hist"]
    w_in = workload_inputs("gpt2s_upproj_fwd")
    x, wm = dev_bf16(torch, w_in["x"]), dev_bf16(torch, w_in["w"])
    dy = dev_bf16(torch, lognormal_grad_bf16(2002, (M, N)))
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device="cuda")
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    wst, xst, gst = g.TensorState(H), g.TensorState(H), g.TensorState(H)
    wq, wqT, xq, dyq = u8(K, N), u8(N, K), u8(M, K), u8(M, N)
    y, dx, dw = bf(M, N), bf(M, K), bf(K, N)
    D, T = g.FP8_SCALE_DELAYED, g.FP8_GRAN_TENSOR
    fl = 2.0 * M * N * K
    bwd = [g.mm_problem(xq, 0, dyq, 1, K, N, M, K, N, xst.scale_inv, gst.scale_inv, dw, N, mn_major=1),
           g.mm_problem(dyq, 1, wq, 0, M, K, N, N, N, gst.scale_inv, wst.scale_inv, dx, K)]
    wsb = max(g.fp8_scaled_mm_grouped_workspace_bytes(bwd), g.fp8_scaled_mm_workspace_bytes(M, N, K))
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    stages = [
        Stage("requant_w", lambda: g.fp8_requantize_weights(wm, K, N, T, D, wst, wq, wqT), 1, nbytes=K * N * 4.0),
        Stage("quant_x", lambda: g.fp8_quantize(x, M, K, K, g.FP8_E4M3, T, D, xst, xq, None), 1, nbytes=M * K * 3.0),
        Stage("gemm_fwd", lambda: g.fp8_scaled_mm_ws(xq, 0, wqT, 0, M, N, K, K, K, T, xst.scale_inv, wst.scale_inv,
                                                     y, N, ws, wsb), 1, flops=fl),
        Stage("quant_dy", lambda: g.fp8_quantize(dy, M, N, N, g.FP8_E5M2, T, D, gst, dyq, None), 1, nbytes=M * N * 3.0),
        Stage("gemm_bwd", lambda: g.fp8_scaled_mm_grouped(bwd, ws, wsb), 1, flops=2 * fl),
        Stage("commit", lambda: g.fp8_history_commit_many([wst, xst, gst]), 1),
    ]
    side = torch.cuda.Stream()

    def enqueue():
        side.wait_stream(stream)
        stages[0].fn()
        with torch.cuda.stream(side):
            stages[1].fn()
        stream.wait_stream(side)
        for st in stages[2:]:
            st.fn()

    def reset():
        for s in (wst, xst, gst):
            s.reset()  # the delayed-scaling state starts empty (bootstrap step first)

    step_ms, stage_ms, _ = time_step(torch, stream, flush, enqueue, stages, steps, warmup, before_replays=reset)
    ms = sum(step_ms) / steps
    return {"value": round(3 * fl / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
            "steps": steps,
            "config": {"workload": "gpt2s_upproj_train_step", "M_tokens": M, "d_model": K, "d_ff": N,
                       "scaling": "per-tensor delayed, amax history 16",
                       "step": "(requantise W || quantise x), fwd GEMM, quantise dy, dgrad + wgrad in one grouped "
                               "launch, 3 history commits; one CUDA graph on two streams"},
            "roofline": roofline(stages, stage_ms, ctx["hbm"], ctx["bf16_tf"], ctx["peak_src"]),
            "kernels": kernel_records(stages, stage_ms, ctx["hbm"], ctx["fp8_peak"])}


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
    ("fine_fwd_mx", 16384, 14336, 4096, 0, 0, "mx"),
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
        if blk == "mx":  # UE8M0 scale atoms, exponents in [-7, 7]
            sa = torch.randint(120, 135, (-(-m // 128) * (k // 128) * 512,), generator=gen, device="cuda",
                               dtype=torch.int32).to(torch.uint8)
            sb = torch.randint(120, 135, (-(-n // 128) * (k // 128) * 512,), generator=gen, device="cuda",
                               dtype=torch.int32).to(torch.uint8)
            gran = g.FP8_GRAN_MX_1x32
        elif blk:
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
    xq, dyq = u8(tokens, d), u8(tokens, n)
    y, dx, dw = bf(tokens, n), bf(tokens, d), bf(d, n)
    wsb = g.fp8_linear_bwd_workspace_bytes(tokens, d, n)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    D, T = g.FP8_SCALE_DELAYED, g.FP8_GRAN_TENSOR

    def layer_step(l):  # the layer API: 6 launches (update + requantise, x cast, forward GEMM,
        ws_, xs, gs = st[l]  # dy cast, grouped dgrad + wgrad, history commit)
        g.fp8_update_requantize_weights(W[l], delta[l], d, n, D, ws_, wq[l], wqT[l])
        g.fp8_linear_fwd(x, tokens, d, n, wqT[l], ws_, None, xs, T, D, xq, None, None, y)
        g.fp8_linear_bwd_mn(dy, tokens, d, n, xq, xs, wq[l], ws_, gs, D, dyq, dx, dw, ws, wsb)
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
# Each leg times the oracle (as it stands: numpy, fp64 matmuls through the BLAS) on bounded
# slabs of one workload's step and extrapolates linearly to the full step: the casts are
# per-element work and the GEMM slabs cover a fraction of the output rows (or of the
# contraction), so time scales with the slab. The numpy casts run on one thread; the
# matmuls on as many threads as the BLAS is given.
def _t(fn):
    t0 = time.perf_counter()
    out = fn()
    return time.perf_counter() - t0, out


FINE_SLAB_COLS = 1792  # 14 of the 112 column blocks of W (and of y)


def finegrained_slab(rows: int, cols: int = FINE_SLAB_COLS):
    """The first `rows` rows of the headline's x and the first `cols` columns of its W (the
    workload's own draws)."""
    import numpy as np
    from datagen import workload_inputs
    w_in = workload_inputs("finegrained_fwd", M=rows)  # the first rows of the full x
    return w_in["x"], np.ascontiguousarray(w_in["w"][:, :cols])


def leg_finegrained(rows: int):
    """x's 1x128 cast on `rows` of 16384 rows, W's 128x128 cast on 1792 of 14336 columns, the
    block-scaled GEMM on the rows x 1792 output slab they give."""
    from oracle import fp8, gemm, quant
    M, K, N = FINE["M"], FINE["K"], FINE["N"]
    x, w = finegrained_slab(rows)
    t_x, ox = _t(lambda: quant.quantize_tile_1x128(x, fp8.E4M3))
    t_w, ow = _t(lambda: quant.quantize_block_128x128(w, fp8.E4M3))
    t_g, _ = _t(lambda: gemm.block_scaled_mm(ox["q"], fp8.E4M3, ox["d"], ow["qT"], fp8.E4M3, ow["d"]))
    c = FINE_SLAB_COLS
    parts = {"cast_x_1x128": t_x * M / rows, "cast_w_128x128": t_w * N / c, "gemm_block_scaled": t_g * (M / rows) * (N / c)}
    return 2.0 * M * N * K, parts, (f"x 1x128 cast of {rows} of {M} rows, W 128x128 cast of {c} of {N} columns, "
                                     f"block-scaled GEMM on the {rows} x {c} output slab; extrapolated linearly")


def leg_finegrained_mx(rows: int):
    """The MX casts of `rows` rows of x and 32 columns of W, the MX GEMM on the rows x 32
    output slab they give (the oracle's MX cast visits every group of 32 in Python)."""
    import numpy as np
    from oracle import fp8, gemm, quant
    M, K, N = FINE["M"], FINE["K"], FINE["N"]
    c = 32
    x, w = finegrained_slab(rows, c)
    t_x, ox = _t(lambda: quant.quantize_mx(x, fp8.E4M3))
    t_w, ow = _t(lambda: quant.quantize_mx(np.ascontiguousarray(w.T), fp8.E4M3))
    t_g, _ = _t(lambda: gemm.mx_scaled_mm(ox["q"], fp8.E4M3, ox["e"], ow["q"], fp8.E4M3, ow["e"]))
    parts = {"cast_x_mx": t_x * M / rows, "cast_w_mx": t_w * N / c, "gemm_mx": t_g * (M / rows) * (N / c)}
    return 2.0 * M * N * K, parts, (f"x MX cast of {rows} of {M} rows, W MX cast of {c} of {N} columns, MX GEMM "
                                     f"on the {rows} x {c} output slab; extrapolated linearly")


def leg_backward(rows: int):
    """dy's per-tensor E5M2 cast (current scaling) on `rows` of the 16384 rows; dgrad on `rows`
    output rows; wgrad over `rows` of the 16384 tokens of its contraction."""
    from datagen import normal_bf16, lognormal_grad_bf16
    from oracle import fp8, gemm, quant
    M, K, N = BWD["M"], BWD["K"], BWD["N"]
    base = 3000
    x = normal_bf16(base + 0, (rows, K))                 # the first rows of the workload's x
    w = normal_bf16(base + 1, (K, N), 0.02)
    dy = lognormal_grad_bf16(base + 2, (rows, N))        # the first rows of its dy
    ow = quant.quantize_tensor(w, fp8.E4M3)
    ox = quant.quantize_tensor(x, fp8.E4M3)
    t_c, og = _t(lambda: quant.quantize_tensor(dy, fp8.E5M2))
    t_d, _ = _t(lambda: gemm.scaled_mm(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"]))
    t_w, _ = _t(lambda: gemm.scaled_mm(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"]))
    f = M / rows
    parts = {"cast_dy": t_c * f, "gemm_dgrad": t_d * f, "gemm_wgrad": t_w * f}
    return 2 * 2.0 * M * N * K, parts, (f"dy cast on {rows} of {M} rows, dgrad on {rows} output rows, wgrad over "
                                        f"{rows} of {M} tokens; extrapolated linearly")


def leg_delayed_loop(rows: int):
    """One layer-step with delayed scaling (states after one bootstrap step): the optimizer
    step and W's full cast, x's and dy's casts on `rows` of the 32768 tokens, the forward and
    dgrad on `rows` output rows, wgrad over `rows` tokens of its contraction."""
    from datagen import normal_bf16, lognormal_grad_bf16, perturbation_f32
    from oracle import fp8, gemm, linear, quant
    M, K, N, H = LOOP["M"], LOOP["K"], LOOP["N"], LOOP["hist"]
    base = 5000
    x = normal_bf16(base + 0, (rows, K))
    dy = lognormal_grad_bf16(base + 2, (rows, N))
    w = normal_bf16(base + 100, (K, N), 0.02)
    delta = perturbation_f32(base + 10_000 + 100 + 0, (K, N), 1e-3)
    ws, xs, gs = quant.DelayedState(H), quant.DelayedState(H), quant.DelayedState(H)
    for st, t, f in ((ws, w, fp8.E4M3), (xs, x, fp8.E4M3), (gs, dy, fp8.E5M2)):  # bootstrap step
        st.quantize(t, f)
        st.commit()
    t_w, wo = _t(lambda: ws.quantize(linear.perturb_master(w, delta), fp8.E4M3))
    t_x, xo = _t(lambda: xs.quantize(x, fp8.E4M3))
    t_c, go = _t(lambda: gs.quantize(dy, fp8.E5M2))
    t_f, _ = _t(lambda: gemm.scaled_mm(xo["q"], fp8.E4M3, wo["qT"], fp8.E4M3, xo["d"], wo["d"]))
    t_d, _ = _t(lambda: gemm.scaled_mm(go["q"], fp8.E5M2, wo["q"], fp8.E4M3, go["d"], wo["d"]))
    t_g, _ = _t(lambda: gemm.scaled_mm(xo["qT"], fp8.E4M3, go["qT"], fp8.E5M2, xo["d"], go["d"]))
    f = M / rows
    parts = {"update_cast_w": t_w, "cast_x": t_x * f, "cast_dy": t_c * f, "gemm_fwd": t_f * f,
             "gemm_dgrad": t_d * f, "gemm_wgrad": t_g * f}
    return 3 * 2.0 * M * N * K, parts, (f"one layer-step: W update + cast in full; x, dy casts on {rows} of {M} "
                                        f"tokens; GEMMs on {rows} output rows (wgrad: {rows} tokens of its "
                                        f"contraction); extrapolated linearly")


def leg_gpt2(rows: int):
    """The GPT-2-small step's arithmetic (current scaling) with the GEMMs on `rows` of the
    8192 tokens; W's cast in full."""
    from datagen import outlier_normal_bf16, normal_bf16, lognormal_grad_bf16
    from oracle import fp8, gemm, quant
    M, K, N = GPT2["M"], GPT2["K"], GPT2["N"]
    x = outlier_normal_bf16(2000, (M, K))[:rows]
    w = normal_bf16(2001, (K, N), 0.02)
    dy = lognormal_grad_bf16(2002, (rows, N))
    t_w, ow = _t(lambda: quant.quantize_tensor(w, fp8.E4M3))
    t_x, ox = _t(lambda: quant.quantize_tensor(x, fp8.E4M3))
    t_c, og = _t(lambda: quant.quantize_tensor(dy, fp8.E5M2))
    t_f, _ = _t(lambda: gemm.scaled_mm(ox["q"], fp8.E4M3, ow["qT"], fp8.E4M3, ox["d"], ow["d"]))
    t_d, _ = _t(lambda: gemm.scaled_mm(og["q"], fp8.E5M2, ow["q"], fp8.E4M3, og["d"], ow["d"]))
    t_g, _ = _t(lambda: gemm.scaled_mm(ox["qT"], fp8.E4M3, og["qT"], fp8.E5M2, ox["d"], og["d"]))
    f = M / rows
    parts = {"cast_w": t_w, "cast_x": t_x * f, "cast_dy": t_c * f, "gemm_fwd": t_f * f, "gemm_dgrad": t_d * f,
             "gemm_wgrad": t_g * f}
    return 3 * 2.0 * M * N * K, parts, (f"W cast in full; x, dy casts and the GEMMs on {rows} of {M} tokens; "
                                        f"extrapolated linearly (current scaling)")


# leg name -> (function, slab rows with all cores, slab rows on one core)
CPU_LEGS = {"finegrained": (leg_finegrained, 1024, 256), "finegrained_upproj_fwd_mx": (leg_finegrained_mx, 128, 32), "backward_upproj": (leg_backward, 1024, 256),
            "delayed_loop": (leg_delayed_loop, 1024, 256), "gpt2s_train_step": (leg_gpt2, 2048, 512)}


def run_cpu_leg(name: str, rows: int):
    fn = CPU_LEGS[name][0]
    t0 = time.perf_counter()
    flops, parts, sample = fn(rows)
    step_s = sum(parts.values())
    return {"value": round(flops / step_s / 1e12, 6), "unit": "TFLOP/s", "step_s_extrapolated": round(step_s, 3),
            "parts_s": {k: round(v, 4) for k, v in parts.items()}, "sample": sample,
            "leg_wall_s": round(time.perf_counter() - t0, 2)}


def cpu_baselines():
    """Every leg twice, in child processes (started before this process uses the GPU): with the
    BLAS on all host cores and on one core."""
    out = {}
    ncpu = os.cpu_count() or 1
    for name, (_, rows_all, rows_one) in CPU_LEGS.items():
        rec = {}
        for threads, rows in ((ncpu, rows_all), (1, rows_one)):
            env = dict(os.environ)
            for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
                env[v] = str(threads)
            env["CUDA_VISIBLE_DEVICES"] = ""
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-leg", name, "--rows", str(rows)],
                               capture_output=True, text=True, env=env, timeout=600)
            try:
                rec[threads] = json.loads(r.stdout.strip().splitlines()[-1])
            except (IndexError, json.JSONDecodeError):
                rec[threads] = {"error": (r.stderr or r.stdout)[-300:]}
        a, o = rec[ncpu], rec[1]
        out[name] = {"value": a.get("value"), "unit": "TFLOP/s", "cores": ncpu, "kind": "oracle",
                     "sample": a.get("sample", "") + f"; numpy casts on one thread, fp64 BLAS matmuls on {ncpu} cores",
                     "step_s_extrapolated": a.get("step_s_extrapolated"), "parts_s": a.get("parts_s"),
                     "one_core": {"value": o.get("value"), "cores": 1, "sample": o.get("sample"),
                                  "step_s_extrapolated": o.get("step_s_extrapolated")}}
    return out


def run_reference(args):
    """The reference arm: the oracle on a bounded sample of the headline step per timed step
    (x's 1x128 cast on 64 rows, W's 128x128 cast on 1792 columns, the block-scaled GEMM on the
    64 x 1792 output slab), on the host cores; value = the GEMM FLOPs the sample covers per
    second."""
    rank, _, world = env_rank()
    if rank != 0:
        return
    from oracle import fp8, gemm, quant
    M, K, N = FINE["M"], FINE["K"], FINE["N"]
    rows, cols = 64, FINE_SLAB_COLS
    x, w = finegrained_slab(rows)

    def step():
        ox = quant.quantize_tile_1x128(x, fp8.E4M3)
        ow = quant.quantize_block_128x128(w, fp8.E4M3)
        gemm.block_scaled_mm(ox["q"], fp8.E4M3, ox["d"], ow["qT"], fp8.E4M3, ow["d"])
        return 2.0 * rows * cols * K

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    fl = sum(step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    sample = (f"per step: x 1x128 cast of {rows} of {M} rows, W 128x128 cast of {cols} of {N} columns, block-scaled "
              f"GEMM on the {rows} x {cols} output slab; numpy oracle (casts on one thread), fp64 BLAS matmuls "
              f"on all cores")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": "finegrained_upproj_fwd", "M_tokens": M, "d_model": K, "d_ff": N},
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
    ap.add_argument("--headline-only", action="store_true", help="time the headline step only (no sub-records)")
    ap.add_argument("--records", default="", help="comma-separated sub-records to time (default: all of them)")
    ap.add_argument("--sweep", action="store_true", help="time every workload's GEMM and cast shapes instead")
    ap.add_argument("--only", default="", help="comma-separated sweep entries")
    ap.add_argument("--cpu-leg", default="", help=argparse.SUPPRESS)
    ap.add_argument("--rows", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.cpu_leg:
        print(json.dumps(run_cpu_leg(args.cpu_leg, args.rows)))
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
