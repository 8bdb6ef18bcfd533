#!/usr/bin/env python3
"""Benchmark of the FP8_DYNAMIC W8A8 linear layer on one GB300 (per rank).

One *step* is one pass of the whole hot path (per-token quantization, FP8
GEMM, dequant epilogue -- i.e. fp8_linear) over every layer of the workload:
Llama-3.1-8B-shaped decode layers, M in {1, 8, 32} tokens x (K, N) in
{(4096, 6144) QKV, (4096, 4096) O, (4096, 28672) gate/up, (14336, 4096)
down}: 12 fp8_linear calls.  The metric is algorithmic bytes / second
(2MK activations + NK E4M3 weights + 4N weight scales + 2MN outputs per
call).  Weights are rotated over enough sets that their footprint is more
than twice the L2 cache, so every step streams its weights from HBM.

Printed (rank 0, one JSON line): value (device-timed, inputs resident),
e2e (same metric through the public API with pinned host inputs/outputs
copied in the timed region; the step's calls replayed as a CUDA graph, and
issued one by one from Python in e2e.eager), roofline of the dominant kernel (the decode
GEMM), prefill TFLOPS of the 8B prefill shapes as context, the CPU oracle
timed on a bounded sample, and the SM clocks seen during the timed region.

--impl reference times the CPU oracle itself on the same workload.
N > 1 (torchrun): the layer does not shard, so each rank runs an independent
replica; value = all ranks' bytes / the slowest rank's time.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fp8_linear TFLOPS & % FP8 peak (prefill); GB/s & % HBM (decode M≤32)"
WORKLOAD = ("llama-3.1-8b decode linear layers: M in {1,8,32} x (K,N) in "
            "{(4096,6144),(4096,4096),(4096,28672),(14336,4096)}")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor-core ratio (4.5 / 2.25 PFLOP/s)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# Dense FP8 figure for one GB300: NVIDIA's HGX/DGX B300 specifications give
# 72 PFLOPS FP8 per 8 GPUs with 2:4 sparsity, i.e. 4.5 PFLOPS dense per GPU.
NOMINAL_FP8_TFLOPS = 4500.0
NOMINAL_FP8_SOURCE = ("NVIDIA HGX/DGX B300 specifications: 72 PFLOPS FP8 per 8 GPUs with "
                      "2:4 sparsity = 4.5 PFLOPS dense per GPU")
# Dense FP8 tensor-core work per SM per clock (tcgen05.mma kind::f8f6f4),
# measured with an MMA-only loop on every SM (no operand traffic).
FP8_FLOP_PER_CLK_SM = 16384


def config_of(world: int) -> dict:
    """The workload descriptor both arms print (ours and --impl reference)."""
    return {"workload": WORKLOAD,
            "l2_policy": "inputs larger than L2: weights rotated over sets totalling "
                         "more than 2 x L2",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def decode_calls():
    from fp8_w8a8_quantized_gb300 import workloads
    return [(M, K, N) for M in workloads.DECODE_M for (_, K, N) in workloads.SHAPES_8B]


def layer_bytes(M, K, N):
    return 2 * M * K + N * K + 4 * N + 2 * M * N


def gemm_bytes(M, K, N):
    return M * K + 4 * M + N * K + 4 * N + 2 * M * N


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "power_w": statistics.median(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def setup_dist(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(world: int, bytes_per_step: float, steps: int, t_max: float) -> float:
    """Whole-job GB/s of N independent replicas: every rank moves
    bytes_per_step per step; the job takes as long as the slowest rank."""
    return world * bytes_per_step * steps / t_max / 1e9


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_inputs(calls):
    """Host copies of the same synthetic inputs, with the weights quantized
    offline by the oracle (not part of the timed work)."""
    import numpy as np
    import torch

    import oracle
    from fp8_w8a8_quantized_gb300 import workloads
    oracle.build()

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    wcache, items = {}, []
    for (M, K, N) in calls:
        if (K, N) not in wcache:
            w = workloads.weights(N, K, workloads.SEED_DECODE, "cpu")
            wcache[(K, N)] = oracle.quant_rows_bf16(bits(w))
        x = workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, "cpu")
        items.append((M, K, N, bits(x)) + wcache[(K, N)])
    return items


def oracle_step(items):
    import oracle
    for (M, K, N, xb, qw, sw) in items:
        oracle.linear(xb, qw, sw)


def time_oracle(calls, budget_s: float, min_reps: int = 1):
    """Run whole oracle steps until `budget_s` is spent (at least min_reps)."""
    import oracle
    items = oracle_inputs(calls)
    nbytes = sum(layer_bytes(M, K, N) for (M, K, N) in calls)
    reps, t0 = 0, time.perf_counter()
    while reps < min_reps or time.perf_counter() - t0 < budget_s:
        oracle_step(items)
        reps += 1
    dt = time.perf_counter() - t0
    return {"value": nbytes * reps / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "s_per_step": dt / reps, "reps": reps}


def run_reference(args):
    world, rank, _ = setup_dist(args)
    if rank != 0:
        return 0
    calls = decode_calls()
    import oracle
    all_items = oracle_inputs(calls)
    # bounded sample: the longest prefix of the step's calls whose oracle time
    # keeps the whole run (warmup + steps) within about two minutes
    per_call = []
    for it in all_items:
        t0 = time.perf_counter()
        oracle_step([it])
        per_call.append(time.perf_counter() - t0)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n, acc = 0, 0.0
    while n < len(all_items) and (n == 0 or acc + per_call[n] <= budget):
        acc += per_call[n]
        n += 1
    items = all_items[:n]
    sample = ("the whole step (all 12 layer calls)" if n == len(all_items) else
              f"the first {n} of the step's 12 layer calls (M, K, N) = "
              f"{[c[:3] for c in items]}")
    nbytes = sum(layer_bytes(M, K, N) for (M, K, N, *_rest) in items)
    for _ in range(args.warmup):
        oracle_step(items)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(items)
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64 (exact E4M3 products) + f64 epilogue",
        "data": "synthetic", "config": config_of(args.gpus),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch

    import fp8_w8a8_quantized_gb300 as pkg
    from fp8_w8a8_quantized_gb300 import build, workloads

    world, rank, local = setup_dist(args)
    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    pk, pk_kind = peaks()
    calls = decode_calls()

    # weights: rotate enough sets that the footprint exceeds 2 x L2
    per_set = sum(N * K for (_, K, N) in workloads.SHAPES_8B)
    nsets = max(2, -(-2 * l2 // per_set) + 1)
    wsets = []
    for s in range(nsets):
        d = {}
        for (_, K, N) in workloads.SHAPES_8B:
            w = workloads.weights(N, K, workloads.SEED_DECODE + 100 * s, dev)
            d[(K, N)] = pkg.fp8_quant_per_channel_weights(w)
            del w
        wsets.append(d)
    xs = [workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, dev) for (M, K, N) in calls]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (M, K, N) in calls]
    wss = [torch.empty(pkg.fp8_linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
           for (M, K, N) in calls]
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(dev)
    nbytes_step = sum(layer_bytes(M, K, N) for (M, K, N) in calls)

    def step_linear(wset, s):
        for i, (M, K, N) in enumerate(calls):
            wq, sw = wset[(K, N)]
            pkg.fp8_linear(xs[i], wq, sw, y=ys[i], workspace=wss[i], stream=s)

    # one CUDA graph per weight set: a step is one replay
    graphs = []
    with torch.cuda.stream(stream):
        for wset in wsets:
            step_linear(wset, stream)  # warm (per-device setup happens here)
        stream.synchronize()
        for wset in wsets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step_linear(wset, torch.cuda.current_stream())
            graphs.append(g)
    torch.cuda.synchronize()

    def timed(fn_step, steps, warmup):
        with torch.cuda.stream(stream):
            for i in range(warmup):
                fn_step(i)
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(steps):
                fn_step(i)
            e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1e3

    def replay_times(fn_step, n, warmup):
        """Seconds of each of n steps: one event pair per step (consecutive
        events on the launching stream), after `warmup` untimed steps."""
        with torch.cuda.stream(stream):
            for i in range(warmup):
                fn_step(i)
        stream.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(n):
                fn_step(i)
                ev[i + 1].record(stream)
        ev[-1].synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(n)]

    replay = lambda i: graphs[i % nsets].replay()
    with ClockSampler(local) as clk:
        t_main = timed(replay, args.steps, max(args.warmup, 3))
        # the survey's procedure beside the mean: the median of >= 20 graph
        # replays, one event pair per replay (a separate pass)
        per_replay = replay_times(replay, max(20, min(args.steps, 100)), 3)
    t_main = max_over_ranks(t_main, world)
    value = replica_value(world, nbytes_step, args.steps, t_main)
    t_med = max_over_ranks(statistics.median(per_replay), world)
    replays = {"n": len(per_replay), "median_ms_per_step": t_med * 1e3,
               "value_at_median": replica_value(world, nbytes_step, 1, t_med),
               "min_ms_per_step": min(per_replay) * 1e3,
               "max_ms_per_step": max(per_replay) * 1e3,
               "how": "one CUDA-event pair per graph replay (one decode step), separate "
                      "pass after the timed region"}

    # --- dominant kernel alone: the decode GEMM over the same 12 shapes ----
    qx = [pkg.fp8_quant_per_token(x) for x in xs]
    gemm_graphs = []
    with torch.cuda.stream(stream):
        for wset in wsets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i, (M, K, N) in enumerate(calls):
                    wq, sw = wset[(K, N)]
                    pkg.fp8_scaled_gemm(qx[i][0], qx[i][1], wq, sw, y=ys[i],
                                        stream=torch.cuda.current_stream())
            gemm_graphs.append(g)
    gsteps = max(args.steps, 50)
    t_gemm = timed(lambda i: gemm_graphs[i % nsets].replay(), gsteps, 3)
    gbytes = sum(gemm_bytes(M, K, N) for (M, K, N) in calls)
    achieved = gbytes * gsteps / t_gemm / 1e9
    hbm_peak = pk["hbm_gbs"]
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak,
                "traffic": (None if GEMM_DECODE_TRAFFIC_RATIO is None else
                            GEMM_DECODE_TRAFFIC_RATIO * gbytes / len(calls)),
                "bytes_per_launch": gbytes / len(calls),
                "kernel": "gemm_decode_kernel", "peak_kind": f"{pk_kind} copy bandwidth",
                "frac_of_8tbs_spec": achieved / 8000.0}

    # --- prefill context: 8B shapes at M = 2048, 8192 (TFLOPS) -------------
    pre_calls = [(M, K, N) for M in workloads.PREFILL_M for (_, K, N) in workloads.SHAPES_8B]
    pxs = {}
    for (M, K, N) in pre_calls:
        if (M, K) not in pxs:
            pxs[(M, K)] = workloads.student_t_outliers(M, K, workloads.SEED_PREFILL, dev)
    pys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (M, K, N) in pre_calls]
    pws = torch.empty(max(pkg.fp8_linear_workspace_size(M, N, K) for (M, K, N) in pre_calls),
                      dtype=torch.uint8, device=dev)
    wset0 = wsets[0]

    def prefill_step(i):
        for j, (M, K, N) in enumerate(pre_calls):
            wq, sw = wset0[(K, N)]
            pkg.fp8_linear(pxs[(M, K)], wq, sw, y=pys[j], workspace=pws, stream=stream)

    psteps = max(3, min(args.steps, 20))
    with ClockSampler(local) as pclk:
        t_pre = timed(prefill_step, psteps, 2)
    flops = sum(2 * M * N * K for (M, K, N) in pre_calls)
    tflops = flops * psteps / t_pre / 1e12
    fp8_peak = FP8_PER_BF16 * pk["bf16_tflops_sustained"]
    prefill = {"tflops": tflops, "peak_tflops": fp8_peak,
               "peak_kind": f"2 x {pk_kind} sustained bf16 (nominal fp8/bf16 ratio)",
               "frac": tflops / fp8_peak, "frac_of_4500_nominal": tflops / 4500.0,
               "nominal_dense_fp8_tflops": NOMINAL_FP8_TFLOPS,
               "nominal_source": NOMINAL_FP8_SOURCE,
               "workload": "llama-3.1-8b prefill layers, M in {2048,8192}, 8 fp8_linear calls"}
    pc = pclk.summary()
    if pc["sm_mhz"]:
        clk_peak = props.multi_processor_count * FP8_FLOP_PER_CLK_SM * pc["sm_mhz"] * 1e6 / 1e12
        prefill.update({"clock_peak_tflops": clk_peak, "frac_of_clock_peak": tflops / clk_peak,
                        "clock_peak_kind": f"{props.multi_processor_count} SMs x "
                                           f"{FP8_FLOP_PER_CLK_SM} dense FP8 FLOP/clk/SM x "
                                           f"median SM clock {pc['sm_mhz']:.0f} MHz "
                                           "during the prefill timing",
                        "sm_mhz_during": pc["sm_mhz"]})
    del pxs, pys, pws

    decode_70b = decode_70b_rates(pkg, workloads, dev, stream, timed, hbm_peak, args.steps, l2)
    prefill_70b = prefill_70b_rate(pkg, workloads, dev, stream, timed, fp8_peak, args.steps)
    mid_batch = mid_batch_rates(pkg, workloads, dev, stream, timed, hbm_peak, args.steps, l2)
    variants = variant_rates(pkg, workloads, dev, stream, timed, hbm_peak, args.steps)
    blockwise = blockwise_rates(pkg, workloads, dev, stream, timed, hbm_peak, fp8_peak,
                                args.steps, l2)

    # --- e2e: public API with pinned host buffers, copies in the timed region.
    # Every step copies its 12 activations host -> device (one copy from one
    # pinned buffer), runs the 12 layers through fp8_linear from Python and
    # copies the 12 outputs back (one copy).  As a serving loop would, the
    # device buffers are double-buffered across steps and the copies run on
    # their own streams: step i+1's upload overlaps step i's layers, and step
    # i's download overlaps step i+1's layers.  The timed region ends after
    # the last step's download.
    x_sizes = [x.numel() for x in xs]
    y_sizes = [y.numel() for y in ys]
    hx_all = torch.cat([x.reshape(-1).cpu() for x in xs]).pin_memory()
    hys = [torch.empty(sum(y_sizes), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx_all = [torch.empty(hx_all.shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    dy_all = [torch.empty(hys[0].shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    dxs, dys = [[], []], [[], []]
    for b in range(2):
        o = 0
        for (M, K, N), nx in zip(calls, x_sizes):
            dxs[b].append(dx_all[b][o:o + nx].view(M, K))
            o += nx
        o = 0
        for (M, K, N), ny in zip(calls, y_sizes):
            dys[b].append(dy_all[b][o:o + ny].view(M, N))
            o += ny
    h2d = hx_all.numel() * hx_all.element_size()
    d2h = hys[0].numel() * hys[0].element_size()
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    wss2 = [wss, [torch.empty_like(w) for w in wss]]

    def layers(b, wset):
        for j, (M, K, N) in enumerate(calls):
            wq, sw = wset[(K, N)]
            pkg.fp8_linear(dxs[b][j], wq, sw, y=dys[b][j], workspace=wss2[b][j], stream=stream)

    # The same 12 calls captured once per device buffer and weight set, as a
    # serving loop replays its decode step: the graph form of the step.
    step_graphs = [[None] * nsets for _ in range(2)]
    with torch.cuda.stream(stream):
        for b in range(2):
            for k in range(nsets):
                layers(b, wsets[k])
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    layers(b, wsets[k])
                step_graphs[b][k] = g
    torch.cuda.synchronize()

    def e2e_step(i, graphed):
        b = i % 2
        # the upload may overwrite dx[b] once step i-2's layers are done
        h2d_s.wait_event(ev_done[b])
        with torch.cuda.stream(h2d_s):
            dx_all[b].copy_(hx_all, non_blocking=True)
            ev_in[b].record(h2d_s)
        stream.wait_event(ev_in[b])
        # the layers may overwrite dy[b] once step i-2's download is done
        stream.wait_event(ev_out[b])
        if graphed:
            step_graphs[b][i % nsets].replay()
        else:
            layers(b, wsets[i % nsets])
        ev_done[b].record(stream)
        d2h_s.wait_event(ev_done[b])
        with torch.cuda.stream(d2h_s):
            hys[b].copy_(dy_all[b], non_blocking=True)
            ev_out[b].record(d2h_s)

    def e2e_timed(steps, warmup, graphed):
        with torch.cuda.stream(stream):
            for i in range(warmup):
                e2e_step(i, graphed)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(steps):
                e2e_step(i, graphed)
            stream.wait_stream(d2h_s)
            e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1e3

    esteps = max(args.steps, 20)
    t_e2e = max_over_ranks(e2e_timed(esteps, 3, True), world)
    t_eager = max_over_ranks(e2e_timed(esteps, 3, False), world)
    e2e = {"value": replica_value(world, nbytes_step, esteps, t_e2e), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "how": "per step: one pinned-host H2D copy of the 12 activations, the step's 12 "
                  "fp8_linear calls (captured once per device buffer and weight set and "
                  "replayed as a CUDA graph, as a serving loop runs its decode step), one D2H "
                  "copy of the 12 outputs; device buffers double-buffered across steps, "
                  "copies on their own streams (step i+1's upload and step i's download "
                  "overlap the layers)",
           "eager": {"value": replica_value(world, nbytes_step, esteps, t_eager),
                     "unit": "GB/s",
                     "how": "the same steps with the 12 fp8_linear calls issued from Python "
                            "every step instead of a graph replay"}}

    if pkg.fp8_device_status() != pkg.FP8_OK:
        raise RuntimeError("a kernel gave up a bounded wait during the benchmark")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cb = time_oracle(calls, budget_s=args.cpu_budget)
        cpu = {"value": cb["value"], "unit": "GB/s", "cores": cb["cores"], "kind": "oracle",
               "sample": f"whole decode step (12 layer calls), {cb['reps']} step(s), "
                         f"{cb['s_per_step']:.2f} s per step"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": t_main / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate)",
            "data": "synthetic",
            "config": config_of(world),
            "weights": {"sets": nsets, "bytes_per_set": per_set,
                        "rotated_mib": nsets * per_set / 2 ** 20},
            "frac_of_hbm": value / hbm_peak, "frac_of_8tbs_spec": value / 8000.0,
            "replays": replays,
            "gpu_launches": 2 * len(calls) * args.steps,
            "roofline": roofline,
            "prefill": prefill,
            "scale_variants": variants,
            "decode_70b": decode_70b,
            "prefill_70b": prefill_70b,
            "mid_batch": mid_batch,
            "blockwise": blockwise,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    return 0


def blockwise_layer_bytes(M, K, N):
    """Algorithmic bytes of a block-scaled decode layer: bf16 X in, E4M3 W and
    its 128x128 block scales, bf16 Y out."""
    kb, nb = -(-K // 128), -(-N // 128)
    return 2 * M * K + N * K + 4 * nb * kb + 2 * M * N


def blockwise_rates(pkg, workloads, dev, stream, timed, hbm_peak, fp8_peak, steps, l2):
    """The block-scaled layer (1x128 activation groups, 128x128 weight blocks)
    on the same decode step (CUDA graph per weight set, sets > 2 x L2) and the
    same prefill layers as the per-channel path."""
    import torch

    calls = decode_calls()
    per_set = sum(N * K for (_, K, N) in workloads.SHAPES_8B)
    nsets = max(2, -(-2 * l2 // per_set) + 1)
    wsets = []
    for s_ in range(nsets):
        d = {}
        for (_, K, N) in workloads.SHAPES_8B:
            w = workloads.weights(N, K, workloads.SEED_DECODE + 100 * s_, dev)
            d[(K, N)] = pkg.fp8_quant_weight_blocks(w)
            del w
        wsets.append(d)
    xs = [workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, dev) for (M, K, N) in calls]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (M, K, N) in calls]
    wss = [torch.empty(pkg.fp8_linear_blockwise_workspace_size(M, N, K), dtype=torch.uint8,
                       device=dev) for (M, K, N) in calls]
    torch.cuda.synchronize()

    def step(wset, st):
        for i, (M, K, N) in enumerate(calls):
            wq, sw = wset[(K, N)]
            pkg.fp8_linear_blockwise(xs[i], wq, sw, y=ys[i], workspace=wss[i], stream=st)

    graphs = []
    with torch.cuda.stream(stream):
        for wset in wsets:
            step(wset, stream)
        stream.synchronize()
        for wset in wsets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(wset, torch.cuda.current_stream())
            graphs.append(g)
    torch.cuda.synchronize()
    n = max(steps, 50)
    t = timed(lambda i: graphs[i % nsets].replay(), n, 3)
    nbytes = sum(blockwise_layer_bytes(M, K, N) for (M, K, N) in calls)
    gbs = nbytes * n / t / 1e9
    decode = {"gbs": gbs, "frac": gbs / hbm_peak, "ms_per_step": t / n * 1e3,
              "workload": "the decode step above (12 fp8_linear_blockwise calls)"}
    del graphs, xs, ys, wss

    pre_calls = [(M, K, N) for M in workloads.PREFILL_M for (_, K, N) in workloads.SHAPES_8B]
    pxs = {}
    for (M, K, N) in pre_calls:
        if (M, K) not in pxs:
            pxs[(M, K)] = workloads.student_t_outliers(M, K, workloads.SEED_PREFILL, dev)
    pys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (M, K, N) in pre_calls]
    pws = torch.empty(max(pkg.fp8_linear_blockwise_workspace_size(M, N, K)
                          for (M, K, N) in pre_calls), dtype=torch.uint8, device=dev)

    def prefill_step(i):
        for j, (M, K, N) in enumerate(pre_calls):
            wq, sw = wsets[0][(K, N)]
            pkg.fp8_linear_blockwise(pxs[(M, K)], wq, sw, y=pys[j], workspace=pws, stream=stream)

    psteps = max(3, min(steps, 20))
    t = timed(prefill_step, psteps, 2)
    tflops = sum(2 * M * N * K for (M, K, N) in pre_calls) * psteps / t / 1e12
    prefill = {"tflops": tflops, "frac": tflops / fp8_peak,
               "workload": "llama-3.1-8b prefill layers, M in {2048,8192}, 8 calls"}
    del pxs, pys, pws, wsets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return {"decode": decode, "prefill": prefill,
            "launches_per_decode_step": 2 * len(calls)}


def prefill_70b_rate(pkg, workloads, dev, stream, timed, fp8_peak, steps):
    """The 70B-shaped layers at 4096 tokens (config 4's prefill batch): one
    step = 4 fp8_linear calls (QKV, O, gate/up, down), TFLOPS."""
    import torch

    calls = [(4096, K, N) for (_, K, N) in workloads.SHAPES_70B]
    ws_ = {}
    for (_, K, N) in workloads.SHAPES_70B:
        w = workloads.weights(N, K, workloads.SEED_70B, dev)
        ws_[(K, N)] = pkg.fp8_quant_per_channel_weights(w)
        del w
    xs = {}
    for (M, K, N) in calls:
        if (M, K) not in xs:
            xs[(M, K)] = workloads.gaussian_outliers(M, K, workloads.SEED_70B, dev)
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (M, K, N) in calls]
    wsp = torch.empty(max(pkg.fp8_linear_workspace_size(M, N, K) for (M, K, N) in calls),
                      dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def step(i):
        for j, (M, K, N) in enumerate(calls):
            wq, sw = ws_[(K, N)]
            pkg.fp8_linear(xs[(M, K)], wq, sw, y=ys[j], workspace=wsp, stream=stream)

    n = max(3, min(steps, 10))
    t = timed(step, n, 2)
    tflops = sum(2 * M * N * K for (M, K, N) in calls) * n / t / 1e12
    del xs, ys, wsp, ws_
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return {"tflops": tflops, "frac": tflops / fp8_peak, "frac_of_4500_nominal": tflops / 4500.0,
            "workload": "llama-3.1-70b layers at 4096 tokens: (K,N) in {(8192,10240),(8192,8192),"
                        "(8192,57344),(28672,8192)}, 4 fp8_linear calls per step"}


def decode_70b_rates(pkg, workloads, dev, stream, timed, hbm_peak, steps, l2):
    """The 70B-shaped decode layers (32 tokens; QKV, O, gate/up, down: 68 to
    470 MB of E4M3 weights each), one step = 4 fp8_linear calls in a CUDA
    graph, weights rotated over two sets (1.7 GB > 2 x L2)."""
    import torch

    calls = [(32, K, N) for (_, K, N) in workloads.SHAPES_70B]
    per_set = sum(N * K for (_, K, N) in workloads.SHAPES_70B)
    nsets = max(2, -(-2 * l2 // per_set) + 1)
    wsets = []
    for s_ in range(nsets):
        d = {}
        for (_, K, N) in workloads.SHAPES_70B:
            w = workloads.weights(N, K, workloads.SEED_70B + 100 * s_, dev)
            d[(K, N)] = pkg.fp8_quant_per_channel_weights(w)
            del w
        wsets.append(d)
    xs = [workloads.gaussian_outliers(M, K, workloads.SEED_70B, dev) for (M, K, N) in calls]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (M, K, N) in calls]
    wss = [torch.empty(pkg.fp8_linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
           for (M, K, N) in calls]
    torch.cuda.synchronize()

    def step(wset, st):
        for i, (M, K, N) in enumerate(calls):
            wq, sw = wset[(K, N)]
            pkg.fp8_linear(xs[i], wq, sw, y=ys[i], workspace=wss[i], stream=st)

    graphs = []
    with torch.cuda.stream(stream):
        for wset in wsets:
            step(wset, stream)
        stream.synchronize()
        for wset in wsets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(wset, torch.cuda.current_stream())
            graphs.append(g)
    torch.cuda.synchronize()
    n = max(steps, 50)
    t = timed(lambda i: graphs[i % nsets].replay(), n, 3)
    nbytes = sum(layer_bytes(M, K, N) for (M, K, N) in calls)
    gbs = nbytes * n / t / 1e9
    del graphs, xs, ys, wss, wsets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return {"gbs": gbs, "frac": gbs / hbm_peak, "ms_per_step": t / n * 1e3,
            "bytes_per_step": nbytes,
            "workload": "llama-3.1-70b decode linear layers at 32 tokens: (K,N) in "
                        "{(8192,10240),(8192,8192),(8192,57344),(28672,8192)}, 4 fp8_linear "
                        "calls per step"}


def mid_batch_rates(pkg, workloads, dev, stream, timed, hbm_peak, steps, l2):
    """The 8B layers at 128 and 256 tokens (serving batches between the decode
    and prefill configurations; the weight-streaming GEMM with 128- and
    256-token tiles): one step = 8 fp8_linear calls in a CUDA graph, weights
    rotated over sets larger than L2 in total.  TFLOPS and GB/s (context:
    neither is a configuration the targets name)."""
    import torch

    calls = [(M, K, N) for M in (128, 256) for (_, K, N) in workloads.SHAPES_8B]
    per_set = sum(N * K for (_, K, N) in workloads.SHAPES_8B)
    nsets = max(2, -(-2 * l2 // per_set) + 1)
    wsets = []
    for s_ in range(nsets):
        d = {}
        for (_, K, N) in workloads.SHAPES_8B:
            w = workloads.weights(N, K, 1 + 100 * s_, dev)
            d[(K, N)] = pkg.fp8_quant_per_channel_weights(w)
            del w
        wsets.append(d)
    xs = [workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, dev) for (M, K, N) in calls]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (M, K, N) in calls]
    wss = [torch.empty(pkg.fp8_linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
           for (M, K, N) in calls]
    torch.cuda.synchronize()

    def step(wset, st):
        for i, (M, K, N) in enumerate(calls):
            wq, sw = wset[(K, N)]
            pkg.fp8_linear(xs[i], wq, sw, y=ys[i], workspace=wss[i], stream=st)

    graphs = []
    with torch.cuda.stream(stream):
        for wset in wsets:
            step(wset, stream)
        stream.synchronize()
        for wset in wsets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(wset, torch.cuda.current_stream())
            graphs.append(g)
    torch.cuda.synchronize()
    n = max(steps, 50)
    t = timed(lambda i: graphs[i % nsets].replay(), n, 3)
    nbytes = sum(layer_bytes(M, K, N) for (M, K, N) in calls)
    flops = sum(2 * M * N * K for (M, K, N) in calls)
    gbs = nbytes * n / t / 1e9
    del graphs, xs, ys, wss, wsets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return {"tflops": flops * n / t / 1e12, "gbs": gbs, "frac_of_hbm": gbs / hbm_peak,
            "ms_per_step": t / n * 1e3,
            "workload": "llama-3.1-8b linear layers at M in {128, 256}: 8 fp8_linear calls "
                        "per step"}


def variant_rates(pkg, workloads, dev, stream, timed, hbm_peak, steps):
    """GB/s of the quantizers with other scale granularities, each on inputs
    rotated over buffers larger than L2 in total.  Algorithmic bytes: bf16
    read once, E4M3 written once (plus the fp32 per-row scales / slot ids)."""
    import torch

    out = {}
    M, K, nbuf = 8192, 4096, 4           # 8B prefill chunk entering q/k/v or gate/up
    xs = [workloads.student_t_outliers(M, K, workloads.SEED_PREFILL + i, dev)
          for i in range(nbuf)]
    qs = [torch.empty((M, K), dtype=torch.uint8, device=dev) for _ in range(nbuf)]
    s_rows = torch.empty(M, dtype=torch.float32, device=dev)
    s_static = torch.tensor([0.05], dtype=torch.float32, device=dev)
    s_out = torch.empty(1, dtype=torch.float32, device=dev)
    ws = torch.empty(int(pkg.lib().fp8_quant_per_tensor_workspace_size(M, K)),
                     dtype=torch.uint8, device=dev)
    n = max(steps, 40)
    act_bytes = 3 * M * K + 4 * M

    def rate(seconds, nbytes):
        gbs = nbytes * n / seconds / 1e9
        return {"gbs": gbs, "frac": gbs / hbm_peak, "us_per_launch": seconds / n * 1e6}

    def graphed(fn_step, per_graph):
        """Capture per_graph consecutive calls (inputs rotating) in one CUDA
        graph and time n // per_graph replays, so that a short kernel is
        timed on the device rather than at the host's call rate; returns the
        seconds of n calls."""
        with torch.cuda.stream(stream):
            for i in range(per_graph):
                fn_step(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(per_graph):
                fn_step(i)
        reps = max(1, n // per_graph)
        return timed(lambda i: g.replay(), reps, 3) * n / (reps * per_graph)

    t = graphed(lambda i: pkg.fp8_quant_per_token(xs[i % nbuf], xq=qs[i % nbuf], s_tok=s_rows,
                                                  stream=stream), 2 * nbuf)
    out["per_token"] = dict(rate(t, act_bytes), workload=f"{M}x{K} bf16", launches=1)
    t = graphed(lambda i: pkg.fp8_quant_static(xs[i % nbuf], s_static, xq=qs[i % nbuf],
                                               s_rows=s_rows, stream=stream), 2 * nbuf)
    out["static"] = dict(rate(t, act_bytes), workload=f"{M}x{K} bf16", launches=1)
    t = graphed(lambda i: pkg.fp8_quant_per_tensor(xs[i % nbuf], xq=qs[i % nbuf], s=s_out,
                                                   s_rows=s_rows, workspace=ws, stream=stream),
                2 * nbuf)
    out["per_tensor"] = dict(rate(t, act_bytes), workload=f"{M}x{K} bf16", launches=2,
                             note="two passes over x; the second reads it back from the end, "
                                  "partly from L2")
    # RMSNorm with the quantizer fused in, against RMSNorm written to bf16
    # (torch, a library kernel: context only) followed by the quantizer
    gam = (1.0 + 0.1 * torch.randn(K, device=dev)).to(torch.bfloat16)
    t = graphed(lambda i: pkg.fp8_rmsnorm_quant(xs[i % nbuf], gam, 1e-6, xq=qs[i % nbuf],
                                                s_tok=s_rows, stream=stream), 2 * nbuf)
    out["rmsnorm_quant"] = dict(rate(t, act_bytes + 2 * K), workload=f"{M}x{K} bf16",
                                launches=1)
    ys = [torch.empty_like(xs[0]) for _ in range(nbuf)]

    def unfused(i):
        ys[i % nbuf] = torch.nn.functional.rms_norm(xs[i % nbuf], (K,), gam, 1e-6)
        pkg.fp8_quant_per_token(ys[i % nbuf], xq=qs[i % nbuf], s_tok=s_rows, stream=stream)

    t2 = graphed(unfused, 2 * nbuf)
    out["rmsnorm_quant"]["unfused_us_per_call"] = t2 / n * 1e6
    out["rmsnorm_quant"]["unfused"] = "torch rms_norm to bf16, then fp8_quant_per_token"
    del xs, qs, ys

    # KV-cache write: 8 KV heads x 128, one layer's keys (or values) of an
    # 8192-token prefill scattered into a paged cache, 16 layers rotated
    T, H, D, nl = 8192, 8, 128, 16
    n_slots = T + 1024
    kvs = [workloads.student_t_outliers(T * H, D, workloads.SEED_PREFILL + 10 + i, dev)
           .view(T, H, D) for i in range(nl)]
    caches = [torch.zeros((n_slots, H, D), dtype=torch.uint8, device=dev) for _ in range(nl)]
    g = torch.Generator(device="cpu")
    g.manual_seed(7)
    slots = torch.randperm(n_slots, generator=g)[:T].to(torch.int64).to(dev)
    kv_scale = torch.linspace(0.25, 2.0, H, dtype=torch.float32, device=dev)
    t = graphed(lambda i: pkg.fp8_kv_cache_quant(kvs[i % nl], kv_scale, caches[i % nl], slots,
                                                 stream=stream), nl)
    out["kv_cache_write"] = dict(rate(t, 3 * T * H * D + 8 * T),
                                 workload=f"T={T} H={H} D={D}, per-head scales, paged slots",
                                 launches=1)
    # the same layer's keys and values in one launch (pairs of the tensors above)
    t = graphed(lambda i: pkg.fp8_kv_cache_quant_kv(
        kvs[2 * i % nl], kvs[(2 * i + 1) % nl], kv_scale, kv_scale, caches[2 * i % nl],
        caches[(2 * i + 1) % nl], slots, stream=stream), nl // 2)
    out["kv_cache_write_kv"] = dict(rate(t, 6 * T * H * D + 8 * T),
                                    workload=f"T={T} H={H} D={D}, keys and values, per-head "
                                             f"scales, paged slots", launches=1)
    del kvs, caches
    torch.cuda.synchronize()
    return out


# DRAM traffic of the decode GEMM relative to its algorithmic bytes, from an
# ncu capture of the current kernel build on a 32 x 8192 -> 28672 layer
# (dram__bytes_read.sum + dram__bytes_write.sum = 238.20 MB against
# 237.09 MB algorithmic).  Traffic
# grows with the bytes streamed, so the per-launch figure is this ratio times
# the mean algorithmic bytes per launch.  None whenever the kernel has
# changed since the capture.
GEMM_DECODE_TRAFFIC_RATIO = (235.326464 + 2.875648) / 237.092992


def run_case(spec: str, reps: int = 4):
    """fp8_linear on one layer (M,K,N) `reps` times: a small, self-contained
    command for profiler captures."""
    import torch

    import fp8_w8a8_quantized_gb300 as pkg
    from fp8_w8a8_quantized_gb300 import build, workloads
    build.build()
    dev = torch.device("cuda", 0)
    kind, *dims = spec.split(",")
    if kind in ("static", "tensor", "kv", "kvkv", "norm"):
        return run_variant_case(pkg, workloads, dev, kind, [int(v) for v in dims], reps)
    if kind == "block":
        M, K, N = (int(v) for v in dims)
        w = workloads.weights(N, K, workloads.SEED_DECODE, dev)
        wq, s_w = pkg.fp8_quant_weight_blocks(w)
        del w
        x = workloads.student_t_outliers(M, K, workloads.SEED_PREFILL, dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(pkg.fp8_linear_blockwise_workspace_size(M, N, K), dtype=torch.uint8,
                         device=dev)
        torch.cuda.synchronize()
        for _ in range(reps):
            pkg.fp8_linear_blockwise(x, wq, s_w, y=y, workspace=ws)
        torch.cuda.synchronize()
        if pkg.fp8_device_status() != pkg.FP8_OK:
            raise RuntimeError("a kernel gave up a bounded wait")
        print(json.dumps({"case": ["block", M, K, N], "reps": reps, "ok": True}))
        return 0
    M, K, N = (int(v) for v in spec.split(","))
    w = workloads.weights(N, K, workloads.SEED_DECODE, dev)
    wq, s_w = pkg.fp8_quant_per_channel_weights(w)
    del w
    x = workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(pkg.fp8_linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    for _ in range(reps):
        pkg.fp8_linear(x, wq, s_w, y=y, workspace=ws)
    torch.cuda.synchronize()
    if pkg.fp8_device_status() != pkg.FP8_OK:
        raise RuntimeError("a kernel gave up a bounded wait")
    print(json.dumps({"case": [M, K, N], "reps": reps, "ok": True}))
    return 0


def run_variant_case(pkg, workloads, dev, kind, dims, reps):
    """static,M,K / tensor,M,K / norm,M,K / kv,T,H,D / kvkv,T,H,D: one
    quantizer variant `reps` times."""
    import torch
    if kind == "norm":
        M, K = dims
        x = workloads.student_t_outliers(M, K, workloads.SEED_PREFILL, dev)
        gam = (1.0 + 0.1 * torch.randn(K, device=dev)).to(torch.bfloat16)
        q = torch.empty((M, K), dtype=torch.uint8, device=dev)
        s_rows = torch.empty(M, dtype=torch.float32, device=dev)
        run = lambda: pkg.fp8_rmsnorm_quant(x, gam, 1e-6, xq=q, s_tok=s_rows)
    elif kind == "kv":
        T, H, D = dims
        kv = workloads.student_t_outliers(T * H, D, workloads.SEED_PREFILL, dev).view(T, H, D)
        cache = torch.zeros((T + 1024, H, D), dtype=torch.uint8, device=dev)
        slots = torch.randperm(T + 1024)[:T].to(torch.int64).to(dev)
        sc = torch.linspace(0.25, 2.0, H, dtype=torch.float32, device=dev)
        run = lambda: pkg.fp8_kv_cache_quant(kv, sc, cache, slots)
    elif kind == "kvkv":
        T, H, D = dims
        k = workloads.student_t_outliers(T * H, D, workloads.SEED_PREFILL, dev).view(T, H, D)
        v = workloads.student_t_outliers(T * H, D, workloads.SEED_PREFILL + 1, dev).view(T, H, D)
        kc = torch.zeros((T + 1024, H, D), dtype=torch.uint8, device=dev)
        vc = torch.zeros((T + 1024, H, D), dtype=torch.uint8, device=dev)
        slots = torch.randperm(T + 1024)[:T].to(torch.int64).to(dev)
        sc = torch.linspace(0.25, 2.0, H, dtype=torch.float32, device=dev)
        run = lambda: pkg.fp8_kv_cache_quant_kv(k, v, sc, sc, kc, vc, slots)
    else:
        M, K = dims
        x = workloads.student_t_outliers(M, K, workloads.SEED_PREFILL, dev)
        q = torch.empty((M, K), dtype=torch.uint8, device=dev)
        s_rows = torch.empty(M, dtype=torch.float32, device=dev)
        if kind == "static":
            s = torch.tensor([0.05], dtype=torch.float32, device=dev)
            run = lambda: pkg.fp8_quant_static(x, s, xq=q, s_rows=s_rows)
        else:
            run = lambda: pkg.fp8_quant_per_tensor(x, xq=q, s_rows=s_rows)
    torch.cuda.synchronize()
    for _ in range(reps):
        run()
    torch.cuda.synchronize()
    print(json.dumps({"case": [kind] + dims, "reps": reps, "ok": True}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--case", default=None,
                    help="M,K,N: run fp8_linear on that one layer a few times and exit; "
                         "static,M,K / tensor,M,K / norm,M,K / kv,T,H,D / kvkv,T,H,D: one "
                         "quantizer variant; "
                         "block,M,K,N: fp8_linear_blockwise on one layer")
    args = ap.parse_args()
    if args.case:
        return run_case(args.case)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
