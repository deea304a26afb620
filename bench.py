#!/usr/bin/env python3
"""Benchmark of the EXL3 linear layer on GB300: GB/s, TFLOP/s and % of roofline vs batch rows.

Workload (default): a q_proj-like layer, K=5120 -> N=12288, 6-bit trellis, mcg
codebook, swept over m = 1, 16, 32, ..., 4096 rows.  One *step* is one pass of
the layer (input rotation + fused GEMM) at every batch size of the sweep.

Roofline per launch (cuda-exl3 README, "Measured"): the layer reads k*n*bits/8
weight bytes and does 2*m*k*n flops; its speed of light is the larger of
bytes / HBM peak and flops / dense fp16 tensor peak (peaks: the measured ones in
MEASURED_PEAKS.json).  ``value`` is the sweep's speed-of-light time divided by
its measured time (summed over GPUs when N > 1), in percent.

Timing: W warm-up steps, then K steps between barrier + synchronize, CUDA events
on the launching stream, max over ranks.  Weights rotate through enough copies
that their total exceeds 3x the 129 MB L2, so every launch reads cold weights.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "EXL3 linear GB/s, TFLOPS and %roofline vs batch rows m=1-4096 (1 GB300)"
UNIT = "% of 1-GPU roofline (sweep SoL time / measured time, summed over GPUs)"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The small-batch call's issue-rate roofline: SMs, maximum SM clock, and the
# warp instructions the column decode spends per 512 decoded values (16 values
# on each of a warp's 32 lanes), counted by ncu on the decode loop alone.
SMS_GB300 = 152
SM_MAX_GHZ = 2.07
DECODE_WARP_INSTR_PER_512 = 104

WORKLOADS = {
    # name: (description, k, shard widths, bits, codebook, m list, split)
    "q_proj_sweep": ("q_proj-like batch sweep: K=5120, N=12288, 6-bit mcg, random trellis, suh/svh sign*U(0.8,1.2), "
                     "x bf16 N(0,1), m=1..4096", 5120, [12288], 6, 1,
                     [1, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096], False),
    "single_4b": ("single linear K=2048, N=4096, 4-bit mcg, m=1,16", 2048, [4096], 4, 1, [1, 16], False),
    "gate_up": ("gate_up K=5120, shards [17408, 17408], 5-bit mul1, m=1,16,128,512", 5120, [17408, 17408], 5, 2,
                [1, 16, 128, 512], False),
    "down_splitk": ("down_proj K=17408, N=5120, 6-bit mul1, split-k, m=1,16,128,512", 17408, [5120], 6, 2,
                    [1, 16, 128, 512], True),
    "lm_head": ("wide head K=4096, N=154880, 6-bit 3inst, m=1,16,512,2048", 4096, [154880], 6, 0,
                [1, 16, 512, 2048], False),
    "proj_12288": ("large projection K=12288, N=4096, 5-bit mcg, m=1,16,512,2048", 12288, [4096], 5, 1,
                   [1, 16, 512, 2048], False),
}


def weight_copies(k, n, bits):
    """Copies of the weights the timed loops rotate over: enough that their total
    exceeds 3x L2, so every launch reads its trellis from HBM."""
    wbytes = k * n * bits // 8
    return max(3, -(-3 * L2_BYTES // wbytes)), wbytes


def workload_config(args, wl_name, world):
    """The config dict of a workload's JSON line (the same for both arms)."""
    desc, k, widths, bits, cb, ms, split = WORKLOADS[wl_name]
    n = sum(widths)
    copies, wbytes = weight_copies(k, n, bits)
    return {"workload": desc, "k": k, "n": n, "bits": bits, "codebook": ["3inst", "mcg", "mul1"][cb],
            "m": ms, "split_k": split, "parallelism": f"replicas x{world} (rows independent)",
            "tile_shape": "autotuned in warm-up" if args.autotune else "cost model",
            "l2": f"weights rotate over {copies} copies ({copies * wbytes / 1e6:.0f} MB > 3x L2)"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"]))}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def sol_seconds(m, k, n, bits, peaks):
    """Speed-of-light time of one linear: max of weight bytes at HBM peak and flops at fp16 peak."""
    t_mem = k * n * bits / 8 / (peaks["hbm_gbs"] * 1e9)
    t_tc = 2.0 * m * k * n / (peaks["bf16_tflops"] * 1e12)
    return max(t_mem, t_tc), ("hbm" if t_mem >= t_tc else "tensor")


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash():
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exl3_trellis_quantized_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def max_over_ranks(value, device):
    """The largest value over the ranks of the process group (the slowest
    replica's time), or the value itself without one; every rank gets it."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(sol_seconds_per_step, steps, world, elapsed):
    """Whole-job % of the 1-GPU roofline: every replica runs `steps` steps of
    the workload, so the job does world * steps of speed-of-light work in the
    slowest replica's time."""
    return 100.0 * sol_seconds_per_step * steps * world / elapsed


def recorded_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel_key)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------


def run_gpu(args, wl_name):
    import torch
    import torch.distributed as dist

    import exl3_trellis_quantized_gb300 as E
    from exl3_trellis_quantized_gb300 import synthetic

    desc, k, widths, bits, cb, ms, split = WORKLOADS[wl_name]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    E.lib()  # fail loudly if the library is missing
    E.set_autotune(args.autotune)  # the tile shapes are tuned in the first warm-up step
    peaks, peak_src = load_peaks()

    layer = synthetic.make_layer(k, widths, bits, cb, seed=1002)
    n = layer.n
    copies, wbytes = weight_copies(k, n, bits)
    assert wbytes == layer.trellis.numel() * 2
    trs = [layer.trellis.to(dev)]
    for _ in range(copies - 1):
        trs.append(trs[0].clone())
    suh = layer.suh.to(dev)
    svh = layer.svh.to(dev)
    mmax = max(ms)
    x_host = synthetic.make_x(mmax, k, seed=1002)
    x_dev = x_host.to(dev)
    xs = [x_dev[:m] for m in ms]
    xh = [torch.empty((len(widths), m, k), dtype=torch.float16, device=dev) for m in ms]
    ys = [torch.empty((m, n), dtype=torch.bfloat16, device=dev) for m in ms]
    accs = [torch.zeros(max(1, E.splitk_workspace_bytes(m, k, n) // 4), dtype=torch.float32, device=dev)
            if split else None for m in ms]
    stream = torch.cuda.current_stream(dev)
    # launches per step: per batch size the transform, the GEMM (two launches
    # when the cost model splits off a pair tile's last wave) and, under
    # split-k, the epilogue
    from exl3_trellis_quantized_gb300 import binding as EB
    launches_per_step = sum(
        2 + (1 if EB.test_tile_plan(m, k, n, layer.shard_cols, split)[1] >= 0 else 0)
        + (1 if split and E.splitk_parts(k, n) > 1 else 0) for m in ms)

    def one_linear(i, it):
        tr = trs[it % copies]
        E.input_transform(xs[i], suh, xh[i])
        if split:
            E.gemm_splitk(xh[i], tr, bits, cb, svh, layer.shard_cols, accs[i], out=ys[i])
        else:
            E.gemm(xh[i], tr, bits, cb, svh, layer.shard_cols, out=ys[i])

    counter = [0]
    # the dominant call: the largest batch, whose GEMM the roofline reports;
    # the small call: m = 16 (else the smallest batch), the HBM-bound regime,
    # reported as roofline_small
    dom = max(range(len(ms)), key=lambda i: ms[i])
    small = ms.index(16) if 16 in ms else min(range(len(ms)), key=lambda i: ms[i])

    def step(events=None, gemm_events=None):
        for i in range(len(ms)):
            if events is not None:
                events[i][0].record(stream)
            if gemm_events is not None and i in gemm_events:
                # events around the GEMM launch(es) alone, on their stream
                tr = trs[counter[0] % copies]
                E.input_transform(xs[i], suh, xh[i])
                gemm_events[i][0].record(stream)
                if split:
                    E.gemm_splitk(xh[i], tr, bits, cb, svh, layer.shard_cols, accs[i], out=ys[i])
                else:
                    E.gemm(xh[i], tr, bits, cb, svh, layer.shard_cols, out=ys[i])
                gemm_events[i][1].record(stream)
            else:
                one_linear(i, counter[0])
            counter[0] += 1
            if events is not None:
                events[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # --- device-resident timed region -------------------------------------
    per_m_ms = [0.0] * len(ms)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    call_ev = [{i: [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
                for i in {dom, small}} for _ in range(args.steps)]
    t0.record(stream)
    for j in range(args.steps):
        step(gemm_events=call_ev[j])
    t1.record(stream)
    torch.cuda.synchronize()
    dom_launch_s = sum(ev[dom][0].elapsed_time(ev[dom][1]) for ev in call_ev) / args.steps / 1e3
    small_launch_s = sum(ev[small][0].elapsed_time(ev[small][1]) for ev in call_ev) / args.steps / 1e3
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, dev)

    # per-batch-size breakdown, measured separately (same launches, events
    # around each; no host synchronisation between steps, so the host stays
    # ahead of the device as in the timed region)
    reps = max(3, min(args.steps, 50))
    per_m_samples = [[] for _ in ms]
    bd_ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in ms]
             for _ in range(reps)]
    for j in range(reps):
        step(bd_ev[j])
    torch.cuda.synchronize()
    for j in range(reps):
        for i in range(len(ms)):
            t_ms = bd_ev[j][i][0].elapsed_time(bd_ev[j][i][1])
            per_m_ms[i] += t_ms
            per_m_samples[i].append(t_ms)
    per_m_s = [v / reps / 1e3 for v in per_m_ms]

    def pct(vals, q):
        v = sorted(vals)
        return v[min(len(v) - 1, int(q * (len(v) - 1) + 0.5))]

    # The same linears replayed from a CUDA graph: `reps` back-to-back linears
    # of one batch size (weights rotating) captured once, so the time excludes
    # host launch overhead (small layers at small m are launch-bound otherwise).
    graph_s = []
    cap_stream = torch.cuda.Stream(dev)
    cap_stream.wait_stream(stream)
    for i in range(len(ms)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(g, stream=cap_stream):
                for r in range(reps):
                    one_linear(i, r + i)
        g.replay()
        torch.cuda.synchronize()
        e0g, e1g = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0g.record(stream)
        for _ in range(3):
            g.replay()
        e1g.record(stream)
        torch.cuda.synchronize()
        graph_s.append(e0g.elapsed_time(e1g) / 1e3 / (3 * reps))
        del g

    # A bandwidth ruler in the same process: a device-to-device copy of 2 GiB.
    # A kernel reading above it flags a timing artefact.
    ruler_src = torch.empty(1 << 30, dtype=torch.int16, device=dev)
    ruler_dst = torch.empty_like(ruler_src)
    ruler_dst.copy_(ruler_src)
    torch.cuda.synchronize()
    er0, er1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    er0.record(stream)
    for _ in range(5):
        ruler_dst.copy_(ruler_src)
    er1.record(stream)
    torch.cuda.synchronize()
    ruler_gbps = 5 * 2 * ruler_src.numel() * 2 / (er0.elapsed_time(er1) / 1e3) / 1e9
    del ruler_src, ruler_dst

    sol_step = sum(sol_seconds(m, k, n, bits, peaks)[0] for m in ms)
    value = replica_throughput(sol_step, args.steps, world, elapsed)

    # Per-batch-size GEMM breakdown: each batch size's GEMM runs `reps` times
    # back to back between two events (weights rotating over the copies, so no
    # launch finds its trellis in L2); a launch's time is the span over `reps`.
    gemm_s = []
    gev = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    for i, m in enumerate(ms):
        E.input_transform(xs[i], suh, xh[i])
        torch.cuda.synchronize()
        gev[0].record(stream)
        for r in range(reps):
            tr = trs[(r + i) % copies]
            if split:
                E.gemm_splitk(xh[i], tr, bits, cb, svh, layer.shard_cols, accs[i], out=ys[i])
            else:
                E.gemm(xh[i], tr, bits, cb, svh, layer.shard_cols, out=ys[i])
        gev[1].record(stream)
        torch.cuda.synchronize()
        gemm_s.append(gev[0].elapsed_time(gev[1]) / 1e3 / reps)
    # The roofline's kernel: the dominant (largest-batch) GEMM call, its average
    # duration taken from the events around it in every step of the timed
    # region (both launches when its last wave is split off).
    md = ms[dom]
    _, bound = sol_seconds(md, k, n, bits, peaks)
    if bound == "hbm":
        achieved = k * n * bits / 8 / dom_launch_s / 1e9
        peak, unit_r = peaks["hbm_gbs"], "GB/s"
    else:
        achieved = 2.0 * md * k * n / dom_launch_s / 1e12
        peak, unit_r = peaks["bf16_tflops"], "TFLOP/s"
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit_r,
                "frac": round(achieved / peak, 4), "peak_source": peak_src + " burst",
                "kernel": f"exl3 GEMM at m={md}", "launch_us": round(dom_launch_s * 1e6, 2),
                "timed": f"CUDA events around the call in each of the {args.steps} timed steps",
                "traffic": recorded_traffic(f"{wl_name}:m={md}")}

    # The HBM-bound regime's kernel: the m = 16 call, against the copy bandwidth.
    ms_small = ms[small]
    achieved_s = k * n * bits / 8 / small_launch_s / 1e9
    roofline_small = {"bound": "hbm", "achieved": round(achieved_s, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": round(achieved_s / peaks["hbm_gbs"], 4), "peak_source": peak_src + " copy bandwidth",
                      "kernel": f"exl3 GEMM at m={ms_small}", "launch_us": round(small_launch_s * 1e6, 2),
                      "timed": f"CUDA events around the call in each of the {args.steps} timed steps",
                      "traffic": recorded_traffic(f"{wl_name}:m={ms_small}")}

    # The same call against the bound of a decode-bound launch: instruction
    # issue.  Peak = 4 warp instructions per cycle per SM x SMs x the maximum
    # SM clock, over the column decode's 104 warp instructions per 512 values
    # (16 values on each of 32 lanes; ncu count of the decode loop alone).
    issue_peak = 4.0 * SMS_GB300 * SM_MAX_GHZ * 1e9
    values_peak = issue_peak * 512.0 / DECODE_WARP_INSTR_PER_512
    values_s = k * n / small_launch_s
    roofline_small_alu = {"bound": "alu", "achieved": round(values_s / 1e9, 1), "peak": round(values_peak / 1e9, 1),
                          "unit": "G decoded values/s", "frac": round(values_s / values_peak, 4),
                          "peak_source": f"issue rate: 4 warp instructions/cycle x {SMS_GB300} SMs x {SM_MAX_GHZ} GHz, "
                                         f"{DECODE_WARP_INSTR_PER_512} warp instructions per 512 decoded values",
                          "kernel": f"exl3 GEMM at m={ms_small}", "launch_us": round(small_launch_s * 1e6, 2)}

    sweep = []
    for i, m in enumerate(ms):
        t = per_m_s[i]
        sol, b = sol_seconds(m, k, n, bits, peaks)
        sweep.append({"m": m, "us": round(t * 1e6, 2), "us_p10": round(pct(per_m_samples[i], 0.1) * 1e3, 2),
                      "us_p90": round(pct(per_m_samples[i], 0.9) * 1e3, 2), "graph_us": round(graph_s[i] * 1e6, 2),
                      "gemm_us": round(gemm_s[i] * 1e6, 2),
                      "GBps": round(k * n * bits / 8 / t / 1e9, 1),
                      "TFLOPS": round(2.0 * m * k * n / t / 1e12, 2),
                      "pct_roofline": round(100.0 * sol / t, 2), "bound": b})

    # --- end to end: pinned host x -> device -> layer -> pinned host y ------
    # Every step copies each batch's x in and its y out.  The copies run on
    # their own streams (one per direction, so both directions overlap each
    # other and the compute), ordered against the compute by events; device x
    # and y are double-buffered so a copy never touches a buffer that a kernel
    # of the other step still uses.
    xpin = [x_host[:m].clone().pin_memory() for m in ms]
    ypin = [torch.empty((m, n), dtype=torch.bfloat16).pin_memory() for m in ms]
    xd2 = [[torch.empty((m, k), dtype=torch.bfloat16, device=dev) for m in ms] for _ in range(2)]
    yd2 = [[torch.empty((m, n), dtype=torch.bfloat16, device=dev) for m in ms] for _ in range(2)]
    h2d = sum(t.numel() * 2 for t in xpin)
    d2h = sum(t.numel() * 2 for t in ypin)
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    x_in = [[ev() for _ in ms] for _ in range(2)]     # x copied in
    x_free = [[ev() for _ in ms] for _ in range(2)]   # transform done with x
    y_done = [[ev() for _ in ms] for _ in range(2)]   # y computed
    y_free = [[ev() for _ in ms] for _ in range(2)]   # y copied out
    used = [[False] * len(ms) for _ in range(2)]

    def e2e_step(it):
        b = it % 2
        for i in range(len(ms)):
            with torch.cuda.stream(h2d_stream):
                if used[b][i]:
                    h2d_stream.wait_event(x_free[b][i])
                xd2[b][i].copy_(xpin[i], non_blocking=True)
                x_in[b][i].record(h2d_stream)
            stream.wait_event(x_in[b][i])
            if used[b][i]:
                stream.wait_event(y_free[b][i])
            tr = trs[(it + i) % copies]
            E.input_transform(xd2[b][i], suh, xh[i])
            x_free[b][i].record(stream)
            if split:
                E.gemm_splitk(xh[i], tr, bits, cb, svh, layer.shard_cols, accs[i], out=yd2[b][i])
            else:
                E.gemm(xh[i], tr, bits, cb, svh, layer.shard_cols, out=yd2[b][i])
            y_done[b][i].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(y_done[b][i])
                ypin[i].copy_(yd2[b][i], non_blocking=True)
                y_free[b][i].record(d2h_stream)
            used[b][i] = True

    def join_copies():
        stream.wait_stream(h2d_stream)
        stream.wait_stream(d2h_stream)

    for w in range(max(1, args.warmup)):
        e2e_step(w)
    join_copies()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_stream.wait_event(e0)
    d2h_stream.wait_event(e0)
    for s in range(args.steps):
        e2e_step(s)
    join_copies()
    e1.record(stream)
    torch.cuda.synchronize()
    e_el = max_over_ranks(e0.elapsed_time(e1) / 1e3, dev)
    e2e_value = replica_throughput(sol_step, args.steps, world, e_el)

    out = None
    if rank == 0:
        cpu = cpu_baseline(wl_name, peaks, budget_s=args.cpu_seconds) if world == 1 and not args.no_cpu else None
        out = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(elapsed / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16 products, fp32 accumulation, bf16 out",
            "data": "synthetic (seeded; random trellis words, sign*U(0.8,1.2) scales, N(0,1) bf16 activations)",
            "config": workload_config(args, wl_name, world),
            "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "roofline": roofline,
            "roofline_small": roofline_small,
            "roofline_small_alu": roofline_small_alu,
            "sweep": sweep,
            "clocks": clk,
            "ruler": {"copy_gbps": round(ruler_gbps, 1), "of_hbm_peak": round(ruler_gbps / peaks["hbm_gbs"], 3)},
            "cpu_baseline": cpu,
            "peaks": {**peaks, "source": peak_src},
        }
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return out


# ---------------------------------------------------------------------------
# CPU oracle arm (baseline only)
# ---------------------------------------------------------------------------


def _cpu_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [p.get("num_threads", 0) for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def _oracle_setup(wl_name):
    from exl3_trellis_quantized_gb300 import synthetic

    desc, k, widths, bits, cb, ms, split = WORKLOADS[wl_name]
    layer = synthetic.make_layer(k, widths, bits, cb, seed=1002)
    x = synthetic.make_x(max(ms), k, seed=1002).float().numpy()
    return layer, x, layer.trellis.numpy(), layer.suh.float().numpy(), layer.svh.float().numpy()


def _oracle_time(setup, m, blocks):
    """Oracle seconds for all m rows of the given 128-column blocks, scaled to the whole layer.

    The oracle's call cost is its input rotation (once per call) plus a part
    per column block; the rotation is timed on its own, and the per-block part
    is scaled by (n/128) / len(blocks).  Returns (scaled seconds, spent seconds).
    """
    from oracle import exl3_oracle as O

    layer, x, tr, suh, svh = setup
    nb = layer.n // 128
    t0 = time.perf_counter()
    O.linear(x[:m], tr, layer.bits, layer.codebook, suh, svh, layer.shard_cols, col_blocks=blocks)
    t1 = time.perf_counter()
    O.input_transform(x[:m], suh)
    t2 = time.perf_counter()
    call, rot = t1 - t0, min(t2 - t1, t1 - t0)
    return rot + (call - rot) * nb / len(blocks), t2 - t0


def cpu_baseline(wl_name, peaks, budget_s=20.0):
    """The FP64 oracle as it stands, timed on a bounded sample of the workload.

    For every batch size of the sweep the oracle computes all m rows of a few
    evenly spaced 128-column blocks; each time is scaled by (n/128) / blocks to
    the whole layer (columns are independent).  Returns the GPU arm's metric.
    """
    import numpy as np

    desc, k, widths, bits, cb, ms, split = WORKLOADS[wl_name]
    setup = _oracle_setup(wl_name)
    n = setup[0].n
    nb = n // 128
    _oracle_time(setup, 1, [0])  # warm-up
    calib = sum(_oracle_time(setup, m, [0])[1] for m in ms)
    per = int(max(1, min(nb, budget_s / max(calib, 1e-3))))
    blocks = sorted(set(int(b) for b in np.linspace(0, nb - 1, per).astype(int)))
    spent = calib
    scaled = 0.0
    for m in ms:
        sc, dt = _oracle_time(setup, m, blocks)
        spent += dt
        scaled += sc
    sol_step = sum(sol_seconds(m, k, n, bits, peaks)[0] for m in ms)
    return {"value": round(100.0 * sol_step / scaled, 6), "unit": UNIT, "cores": _cpu_threads(),
            "kind": "oracle",
            "sample": f"all rows of {len(blocks)} of {nb} 128-column blocks at each m of the sweep; the per-block "
                      f"time scaled by columns to the whole layer ({spent:.1f} s of CPU work)",
            "seconds_per_step_scaled": round(scaled, 3)}


def run_reference(args, wl_name):
    """The oracle arm: each step times the oracle on a bounded sample of the workload.

    A first pass times two 128-column blocks at every batch size of the sweep;
    each timed step then re-times one batch size (rotating through the sweep) on
    two blocks, and the step's sweep time sums, over the batch sizes, the median
    of their samples so far, scaled by columns to the whole layer.
    """
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    peaks, _ = load_peaks()
    desc, k, widths, bits, cb, ms, split = WORKLOADS[wl_name]
    setup = _oracle_setup(wl_name)
    n = setup[0].n
    nb = n // 128
    def blocks_for(i):
        return sorted({(i * 7) % nb, (i * 7 + nb // 2) % nb})

    for m in ms:  # warm-up pass: first calls at each size pay page faults and thread start-up
        _oracle_time(setup, m, blocks_for(0))
    samples = {m: [_oracle_time(setup, m, blocks_for(1))[0]] for m in ms}
    for w in range(args.warmup):
        _oracle_time(setup, ms[w % len(ms)], blocks_for(w + 2))
    latest = {m: statistics.median(v) for m, v in samples.items()}
    sol_step = sum(sol_seconds(m, k, n, bits, peaks)[0] for m in ms)
    vals, steps_s = [], []
    t_all = time.perf_counter()
    for s in range(args.steps):
        m = ms[s % len(ms)]
        samples[m].append(_oracle_time(setup, m, blocks_for(s + 3))[0])
        latest[m] = statistics.median(samples[m])
        step_time = sum(latest.values())
        steps_s.append(step_time)
        vals.append(100.0 * sol_step / step_time)
    el = time.perf_counter() - t_all
    v = round(100.0 * sol_step * len(steps_s) / sum(steps_s), 6) if steps_s else None
    cpu = {"value": v, "unit": UNIT, "cores": _cpu_threads(), "kind": "oracle",
           "sample": f"per step: all m rows of 2 of {nb} 128-column blocks at one batch size of the sweep "
                     f"(rotating); each batch size's time is the median of its samples so far, the per-block "
                     f"part scaled by columns to the layer"}
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, wl_name, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": cpu,
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# Gated MLP block: gate_up GEMM -> SwiGLU folded into the down-projection's
# input transform -> split-k down GEMM (a non-default workload)
# ---------------------------------------------------------------------------
MLP = {"hidden": 5120, "inter": 17408, "gate_up": (5, 2), "down": (6, 2), "m": [1, 16, 128, 512]}


def run_mlp(args):
    import torch

    import exl3_trellis_quantized_gb300 as E
    from exl3_trellis_quantized_gb300 import binding as EB
    from exl3_trellis_quantized_gb300 import synthetic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    E.lib()
    peaks, peak_src = load_peaks()
    hid, inter, ms = MLP["hidden"], MLP["inter"], MLP["m"]
    (gb, gcb), (db, dcb) = MLP["gate_up"], MLP["down"]
    gu = synthetic.make_layer(hid, [inter, inter], gb, gcb, seed=1101)
    dn = synthetic.make_layer(inter, [hid], db, dcb, seed=1102)
    wbytes = (gu.trellis.numel() + dn.trellis.numel()) * 2
    copies = max(3, -(-3 * L2_BYTES // wbytes))
    gtr = [gu.trellis.to(dev)] + [None] * (copies - 1)
    dtr = [dn.trellis.to(dev)] + [None] * (copies - 1)
    for c in range(1, copies):
        gtr[c], dtr[c] = gtr[0].clone(), dtr[0].clone()
    gsuh, gsvh, dsuh, dsvh = gu.suh.to(dev), gu.svh.to(dev), dn.suh.to(dev), dn.svh.to(dev)
    x = synthetic.make_x(max(ms), hid, seed=1103).to(dev)
    bufs = {}
    for m in ms:
        bufs[m] = dict(xh=torch.empty((2, m, hid), dtype=torch.float16, device=dev),
                       g=torch.empty((m, 2 * inter), dtype=torch.bfloat16, device=dev),
                       h=torch.empty((m, inter), dtype=torch.bfloat16, device=dev),
                       dxh=torch.empty((1, m, inter), dtype=torch.float16, device=dev),
                       y=torch.empty((m, hid), dtype=torch.bfloat16, device=dev),
                       acc=torch.zeros(max(1, E.splitk_workspace_bytes(m, inter, hid) // 4), dtype=torch.float32,
                                       device=dev))

    def block(m, it, fused):
        b = bufs[m]
        c = it % copies
        E.input_transform(x[:m], gsuh, b["xh"])
        E.gemm(b["xh"], gtr[c], gb, gcb, gsvh, gu.shard_cols, out=b["g"])
        if fused:
            E.input_transform_swiglu(b["g"], dsuh, b["dxh"])
        else:  # the same step unfused: torch's silu and product, then the plain transform
            torch.mul(torch.nn.functional.silu(b["g"][:, :inter]), b["g"][:, inter:], out=b["h"])
            E.input_transform(b["h"], dsuh, b["dxh"])
        E.gemm_splitk(b["dxh"], dtr[c], db, dcb, dsvh, dn.shard_cols, b["acc"], out=b["y"])

    def timed(fused):
        for w in range(args.warmup):
            for m in ms:
                block(m, w, fused)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for s in range(args.steps):
            for m in ms:
                block(m, s, fused)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / args.steps

    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    t_fused = timed(True)
    clk = clocks.stop()
    t_unfused = timed(False)
    sol = sum(sol_seconds(m, hid, 2 * inter, gb, peaks)[0] + sol_seconds(m, inter, hid, db, peaks)[0] for m in ms)
    return {
        "metric": "EXL3 gated MLP block (gate_up, SwiGLU folded into the down transform, split-k down) %roofline",
        "value": round(100.0 * sol / t_fused, 3), "unit": "% of 1-GPU roofline (both GEMMs' SoL / measured)",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_fused * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16 products, fp32 sums, bf16 out",
        "data": "synthetic (seeded)",
        "config": {"workload": f"gated MLP hidden={hid} inter={inter}, gate_up {gb}-bit mul1 (2 shards), "
                               f"down {db}-bit mul1 split-k, m={ms}",
                   "l2": f"weights rotate over {copies} copies"},
        "unfused_swiglu_ms_per_step": round(t_unfused * 1e3, 4),
        "gpu_launches": sum(
            4 + (1 if E.splitk_parts(inter, hid) > 1 else 0)
            + (1 if EB.test_tile_plan(m, hid, 2 * inter, gu.shard_cols, False)[1] >= 0 else 0)
            + (1 if EB.test_tile_plan(m, inter, hid, dn.shard_cols, True)[1] >= 0 else 0) for m in ms) * args.steps,
        "clocks": clk, "peaks": {**peaks, "source": peak_src},
    }


# ---------------------------------------------------------------------------
# Mixture of experts: gathered per-expert transform + grouped GEMM (non-default)
# ---------------------------------------------------------------------------
MOE = {"hidden": 2048, "inter": 768, "experts": 128, "topk": 8, "bits": 4, "cb": 1, "tokens": [1, 16, 64, 256, 1024]}


def run_moe(args):
    import torch

    import exl3_trellis_quantized_gb300 as E
    from exl3_trellis_quantized_gb300 import synthetic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    E.lib()
    peaks, peak_src = load_peaks()
    hid, inter, ne, topk, bits, cb = (MOE[k] for k in ("hidden", "inter", "experts", "topk", "bits", "cb"))
    n = 2 * inter  # the experts' gate_up layer, two shards
    layer = synthetic.make_moe_layer(hid, [inter, inter], bits, cb, ne, seed=1201)
    expert_bytes = hid * n * bits // 8
    copies = max(3, -(-3 * L2_BYTES // (layer.trellis.numel() * 2)))
    trs = [layer.trellis.to(dev)] + [None] * (copies - 1)
    for c in range(1, copies):
        trs[c] = trs[0].clone()
    suh, svh = layer.suh.to(dev), layer.svh.to(dev)
    runs = []
    for t in MOE["tokens"]:
        # few routed rows per expert: small blocks (16 at about one row per expert,
        # the pages' floor; 32 below 32 rows per expert), else 128
        block = 16 if t * topk <= ne else 32 if t * topk < 32 * ne else 128
        r = synthetic.make_routing(t, ne, topk, block, seed=1202 + t, empty_blocks=0)
        x = synthetic.make_x(t, hid, seed=1203).to(dev)
        ids, be = r.sorted_ids.to(dev), r.block_expert.to(dev)
        xh = torch.empty((2, r.rows, hid), dtype=torch.float16, device=dev)
        y = torch.empty((r.rows, n), dtype=torch.bfloat16, device=dev)
        used = int((r.block_expert >= 0).sum())
        touched = len(set(r.block_expert.tolist()) - {-1})
        runs.append(dict(t=t, block=block, rows=r.rows, x=x, ids=ids, be=be, xh=xh, y=y, blocks=used,
                         bytes=touched * expert_bytes, flops=2.0 * t * topk * hid * n))

    def step(it):
        for run in runs:
            E.moe_input_transform(run["x"], run["ids"], topk, run["be"], run["block"], suh, out=run["xh"])
            E.moe_gemm(run["xh"], trs[it % copies], bits, cb, svh, layer.shard_cols, run["be"], run["block"],
                       out=run["y"])

    for w in range(args.warmup):
        step(w)
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(args.steps):
        step(s)
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    t_step = e0.elapsed_time(e1) / 1e3 / args.steps
    # per-token-count breakdown, measured separately
    per = []
    for run in runs:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        reps = 20
        ev[0].record()
        for i in range(reps):
            E.moe_input_transform(run["x"], run["ids"], topk, run["be"], run["block"], suh, out=run["xh"])
            E.moe_gemm(run["xh"], trs[i % copies], bits, cb, svh, layer.shard_cols, run["be"], run["block"],
                       out=run["y"])
        ev[1].record()
        torch.cuda.synchronize()
        t = ev[0].elapsed_time(ev[1]) / 1e3 / reps
        # the same launches replayed from a CUDA graph (no host launch overhead)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for i in range(reps):
                    E.moe_input_transform(run["x"], run["ids"], topk, run["be"], run["block"], suh, out=run["xh"])
                    E.moe_gemm(run["xh"], trs[i % copies], bits, cb, svh, layer.shard_cols, run["be"],
                               run["block"], out=run["y"])
        g.replay()
        torch.cuda.synchronize()
        ev[0].record()
        for _ in range(3):
            g.replay()
        ev[1].record()
        torch.cuda.synchronize()
        tg = ev[0].elapsed_time(ev[1]) / 1e3 / (3 * reps)
        del g
        # the weighted combine of each token's top-k rows, on rows of the
        # hidden width (the down projection's output), replayed from a graph
        yd = synthetic.make_x(run["rows"], hid, seed=1204).to(dev)
        wt = synthetic.make_topk_weights(run["t"], topk, seed=1205).to(dev)
        table = torch.empty(run["t"] * topk, dtype=torch.int32, device=dev)
        comb = torch.empty((run["t"], hid), dtype=torch.bfloat16, device=dev)
        E.moe_combine(yd, run["ids"], run["be"], run["block"], ne, wt, topk, out=comb, pair_rows=table)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for i in range(reps):
                    E.moe_combine(yd, run["ids"], run["be"], run["block"], ne, wt, topk, out=comb, pair_rows=table)
        g.replay()
        torch.cuda.synchronize()
        ev[0].record()
        for _ in range(3):
            g.replay()
        ev[1].record()
        torch.cuda.synchronize()
        tc = ev[0].elapsed_time(ev[1]) / 1e3 / (3 * reps)
        del g
        comb_bytes = (run["t"] * topk + run["t"]) * hid * 2  # the routed rows read, the combined rows written
        sol = max(run["bytes"] / (peaks["hbm_gbs"] * 1e9), run["flops"] / (peaks["bf16_tflops"] * 1e12))
        per.append({"tokens": run["t"], "block": run["block"], "rows": run["rows"], "live_blocks": run["blocks"],
                    "us": round(t * 1e6, 2), "graph_us": round(tg * 1e6, 2),
                    "GBps_touched_experts": round(run["bytes"] / tg / 1e9, 1),
                    "pct_roofline": round(100.0 * sol / tg, 2),
                    "combine_us": round(tc * 1e6, 2), "combine_GBps": round(comb_bytes / tc / 1e9, 1)})
    sol_step = sum(max(r_["bytes"] / (peaks["hbm_gbs"] * 1e9), r_["flops"] / (peaks["bf16_tflops"] * 1e12))
                   for r_ in runs)
    return {
        "metric": "EXL3 MoE expert gate_up (gathered transform + grouped GEMM) %roofline vs tokens",
        "value": round(100.0 * sol_step / t_step, 3),
        "unit": "% of 1-GPU roofline (touched experts' weight bytes at HBM peak, or routed flops at tensor peak)",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16 products, fp32 sums, bf16 out",
        "data": "synthetic (seeded routing: distinct random top-k experts per token)",
        "config": {"workload": f"{ne} experts, top-{topk}, hidden {hid}, expert gate_up 2x{inter}, {bits}-bit mcg, "
                               f"tokens={MOE['tokens']}", "l2": f"weights rotate over {copies} copies"},
        "sweep": per, "gpu_launches": 2 * len(runs) * args.steps, "clocks": clk,
        "peaks": {**peaks, "source": peak_src},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="q_proj_sweep", choices=sorted(WORKLOADS) + ["mlp_swiglu", "moe"])
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--autotune", action="store_true",
                    help="time every tile shape once per layer shape and batch bucket (in the warm-up)")
    ap.add_argument("--only-m", type=int, default=None,
                    help="restrict the sweep to one batch size (for profiling one launch shape)")
    args = ap.parse_args()
    if args.workload == "moe":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the oracle arm covers the single-layer workloads"}))
            return
        args.warmup = max(args.warmup, 3)
        print(json.dumps(run_moe(args)), flush=True)
        return
    if args.workload == "mlp_swiglu":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the oracle arm covers the single-layer workloads"}))
            return
        args.warmup = max(args.warmup, 3)
        print(json.dumps(run_mlp(args)), flush=True)
        return
    if args.only_m is not None:
        d = list(WORKLOADS[args.workload])
        d[5] = [args.only_m]
        d[0] = d[0] + f" (only m={args.only_m})"
        WORKLOADS[args.workload] = tuple(d)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        out = run_reference(args, args.workload)
    else:
        out = run_gpu(args, args.workload)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
