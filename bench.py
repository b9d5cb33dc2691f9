"""Benchmark of the routed IQ4_NL MoE layer on GB300 (one JSON line on rank 0).

A step is one call of the whole layer (router logits, sigmoid top-k and
weights, per-expert histogram/scan/permutation, gather, dequantising
up/gate + SwiGLU, down projection, weighted combine with the shared expert)
over one batch of synthetic tokens.  Default workload: the Xing4-shaped layer
at decode batch 1 (H 3584, 64 experts top-4 + 1 shared, F 1024, bf16 x).

L2: one layer's working set (~32 MB) fits the 129 MB L2, so steps rotate over
NL resident layers with distinct weights (16 by default: 6.5 GB) and 64
distinct inputs; the data touched in one rotation (16 x 31.9 MB) is about
4x the L2, so each step's weights come from HBM.

Steps run as CUDA-graph replays (G steps per graph) so that the GPU, not
the Python launch loop, sets the pace; the graph holds exactly the launches
of G layer calls.  `e2e` times the same calls eagerly, one
moe_layer_forward_routed_host call per step: the input copied from pinned
host memory, the layer, and the output copied back, enqueued by the library.

--impl reference times the CPU oracle (fp64, single thread) on the same
workload and metric.
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

def expert_bytes_of(wl):
    """IQ4_NL bytes of one expert: up, gate and down, 18 bytes per 32 weights
    (6,193,152 B for the Xing4 layer)."""
    return 3 * wl.F * (wl.H // 32) * 18


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=65536)
    p.add_argument("--warmup", type=int, default=64)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode1",
                   choices=["decode1", "decode8", "decode64", "prefill4096", "trunk38_t1", "trunk38_t16",
                            "k2h_decode1", "k2h_decode64", "k2h_prefill1024"])
    p.add_argument("--layers", type=int, default=16, help="resident layers the steps rotate over")
    p.add_argument("--graph-steps", type=int, default=32)
    p.add_argument("--e2e-steps", type=int, default=2000)
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


METRIC = "MoE-layer tokens/s (expert-weight HBM GB/s as fraction of GB300 peak)"

# DRAM bytes (read + write) per launch of each workload's dominant kernel,
# from the ncu captures summarised in profiles/ (set to None when the kernel
# changes after its capture).
NCU_TRAFFIC = {
    # decode_fused_kernel changed (fewer instructions, the same copies) after
    # its last ncu capture, which read 31,980,544 B per launch: null until it
    # is captured again
    "decode1": None,
    "prefill4096": 457_219_328,   # grouped_gemm_tc<up/gate>, ncu dram read + write per launch
}


def bench_config(args, wl, world):
    T = wl.T
    if wl.n_layers > 1:
        G = max(1, min(args.graph_steps, args.steps, 8))
        return wl.n_layers, 16, G, {
            "workload": wl.name, "tokens_per_step": T, "layers": wl.n_layers, "hidden": wl.H,
            "experts": wl.E, "top_k": wl.k, "expert_ffn": wl.F, "shared_experts": 1,
            "parallelism": f"replicas x{world}",
            "l2": f"{wl.n_layers} resident layers "
                  f"({wl.n_layers * ((wl.E + 1) * expert_bytes_of(wl) + wl.E * wl.H * 4) / 1e9:.1f} GB of weights, "
                  "far larger than L2), 16 rotating inputs",
            "graph_steps": G}
    NL = args.layers if T < 64 else max(1, min(args.layers, 2))
    NX = 64 if T < 64 else 2
    G = max(1, min(args.graph_steps, args.steps))
    return NL, NX, G, {
        "workload": wl.name, "tokens_per_step": T, "hidden": wl.H, "experts": wl.E,
        "top_k": wl.k, "expert_ffn": wl.F, "shared_experts": 1, "routed_scaling": wl.scale,
        "parallelism": f"replicas x{world}",
        "l2": f"rotating over {NL} resident layers and {NX} inputs (inputs larger than L2)",
        "graph_steps": G}


def replay_percentiles(start, marks, per_replay_steps):
    """p10 / median / p90 of the per-step time over the graph replays of the
    timed region (each replay holds per_replay_steps steps), in ms."""
    if not marks:
        return None
    ts, prev = [], start
    for m in marks:
        ts.append(prev.elapsed_time(m) / per_replay_steps)
        prev = m
    ts.sort()
    pick = lambda q: ts[min(len(ts) - 1, int(q * (len(ts) - 1) + 0.5))]
    return {"p10": pick(0.1), "median": pick(0.5), "p90": pick(0.9), "replays": len(ts)}


def algorithmic_bytes(wl, T, distinct_experts):
    """HBM bytes one call must move at least: the selected experts' and the
    shared expert's IQ4_NL weights, the fp32 router, x in and out (bf16)."""
    return (distinct_experts + 1) * expert_bytes_of(wl) + wl.E * wl.H * 4 + 2 * T * wl.H * 2


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [v.strip() for v in ln.split(",")]
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


def cpu_baseline(wl_name, seconds):
    """The oracle as it stands, single-threaded, on a bounded sample of the
    workload: whole tokens through route + forward until `seconds` pass."""
    import numpy as np
    import oracle
    from quantized_moe_expert_sigmoid_gb300 import synth
    wl = synth.WORKLOADS[wl_name]
    ew = synth.expert_weights(0, 0, wl.E, wl.H, wl.F)
    wr = synth.router_weights(0, 0, wl.E, wl.H, wl.router_sigma)
    bias = synth.zipf_logit_bias(0, wl.T, wl.E) if wl.zipf else None
    oracle.build()
    done, t0 = 0, time.perf_counter()
    while True:
        x = oracle.to_f64(synth.activations(0, "bench", 1, wl.H, np.array([done])), "bf16")
        b = None if bias is None else bias[done % wl.T][None, :]
        oracle.moe_layer(x, wr, ew, wl.k, wl.scale, b)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    if wl.n_layers > 1:  # a token crosses every layer of the trunk (plus an RMSNorm each)
        return {"value": done / el / wl.n_layers, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": f"{done} single-token calls of one layer of the {wl_name} trunk "
                          f"({el:.1f} s, fp64, 1 thread), scaled by its {wl.n_layers} layers"}
    return {"value": done / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} single-token layer calls of the {wl_name} workload ({el:.1f} s, fp64, 1 thread)"}


def run_reference(args, rank, world):
    from quantized_moe_expert_sigmoid_gb300 import synth
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    budget = 90.0
    r = cpu_baseline(args.workload, min(budget, 3.0 + 0.2 * (args.steps + args.warmup)))
    _, _, _, cfg = bench_config(args, wl, world)
    line = {"impl": "reference", "metric": METRIC, "value": r["value"],
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "ms_per_step": 1000.0 * wl.T / r["value"],
            "cpu_baseline": r,
            "e2e": {"value": r["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import quantized_moe_expert_sigmoid_gb300 as moe
    from quantized_moe_expert_sigmoid_gb300 import build as moe_build, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(moe_build.LIB):
        moe_build.build()
    if world > 1:
        torch.distributed.barrier()
    wl = synth.WORKLOADS[args.workload]
    T = wl.T
    NL, NX, G, cfg = bench_config(args, wl, world)

    layers, routers = [], []
    for l in range(NL):
        ew = synth.expert_weights_torch(1000 * rank + 7, l, wl.E, wl.H, wl.F, device=dev)
        layers.append(moe.MoeLayer(wl.H, wl.E, wl.k, wl.F, 1, wl.scale, T, up=ew.up, gate=ew.gate,
                                   down=ew.down, sh_up=ew.sh_up, sh_gate=ew.sh_gate,
                                   sh_down=ew.sh_down, flags=moe.MOE_FLAG_HOST_IO))
        del ew
        routers.append(torch.from_numpy(synth.router_weights(7, l, wl.E, wl.H, wl.router_sigma)).to(dev))
    torch.cuda.empty_cache()
    xs_host = [synth.activations(100 + rank, "bench", T, wl.H, np.full(T, i)) for i in range(NX)]
    xs = [torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16) for a in xs_host]
    bias = torch.from_numpy(synth.zipf_logit_bias(7, T, wl.E)).to(dev) if wl.zipf else None
    outs = [torch.empty((T, wl.H), dtype=torch.bfloat16, device=dev) for _ in range(G)]
    ids = [torch.empty((T, wl.k), dtype=torch.int32, device=dev) for _ in range(G)]
    wts = [torch.empty((T, wl.k), dtype=torch.float32, device=dev) for _ in range(G)]

    def step(j, slot):
        L = layers[j % NL]
        moe.moe_layer_forward_routed(L.handle, xs[j % NX], routers[j % NL], ids[slot], wts[slot],
                                     outs[slot], bias)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for j in range(max(3, args.warmup)):
            step(j, j % G)
    stream.synchronize()
    for L in layers:
        L.check()

    # graphs: G steps each; a second graph for a remainder
    def capture(n, offset):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(n):
                step(offset + j, j)
        return g

    reps, rem = divmod(args.steps, G)
    # the batched path has several kernels per call: time its stages with
    # CUDA events recorded inside the graph (event-record nodes refreshed by
    # every replay), so the dominant kernel's own duration is measured in the
    # timed region
    staged = T > 8
    if staged:
        for L in layers:
            moe.moe_layer_enable_timing(L.handle, G)
    launches0 = moe.moe_launch_count()
    g_main = capture(G, 0) if reps else None
    launches_per_graph = moe.moe_launch_count() - launches0
    launches0 = moe.moe_launch_count()
    g_rem = capture(rem, 0) if rem else None
    launches_rem = moe.moe_launch_count() - launches0
    with torch.cuda.stream(stream):
        if g_main:
            g_main.replay()
        if g_rem:
            g_rem.replay()
    stream.synchronize()

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    with Clocks(local_rank) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(reps):
                g_main.replay()
                marks[i].record(stream)
            if g_rem:
                g_rem.replay()
            stop.record(stream)
        stop.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = start.elapsed_time(stop)
    for L in layers:
        L.check()
    t_ms = torch.tensor([ms], device=dev)
    if world > 1:
        torch.distributed.all_reduce(t_ms, op=torch.distributed.ReduceOp.MAX)
    ms = float(t_ms.item())
    steps = reps * G + rem
    stage_ms = None
    if staged:  # per-stage means over the calls of the last replay(s)
        rows = [r for L in layers for r in moe.moe_layer_stage_times(L.handle, G)]
        stage_ms = {name: statistics.fmean(r[i] for r in rows) for i, name in enumerate(moe.STAGES)}
        # the events stay bound to the graphs' nodes: drop both before any
        # eager call on these layers
        del g_main, g_rem
        for L in layers:
            moe.moe_layer_enable_timing(L.handle, 0)
    ms_per_step = ms / steps
    gpu_launches = reps * launches_per_graph + launches_rem

    # distinct experts actually selected per step (for the byte count)
    distinct = []
    for s in range(min(G, steps)):
        distinct.append(len(set(ids[s].flatten().tolist())))
    mean_distinct = sum(distinct) / len(distinct)
    alg_bytes = algorithmic_bytes(wl, T, mean_distinct)
    expert_bytes = (mean_distinct + 1) * expert_bytes_of(wl)

    # end to end through the public API with host buffers
    e2e = None
    if rank == 0:
        n_e2e = max(1, min(args.e2e_steps, args.steps))
        xh = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory() for a in xs_host]
        oh = torch.empty((T, wl.H), dtype=torch.bfloat16).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            # one C-ABI call per step: copy x in, run the layer, copy out back
            for j in range(8):
                moe.moe_layer_forward_routed_host(layers[j % NL].handle, xh[j % NX], routers[j % NL], ids[0],
                                                  wts[0], oh, bias)
            stream.synchronize()
            e0.record(stream)
            for j in range(n_e2e):
                moe.moe_layer_forward_routed_host(layers[j % NL].handle, xh[j % NX], routers[j % NL], ids[0],
                                                  wts[0], oh, bias)
            e1.record(stream)
        e1.synchronize()
        e_ms = e0.elapsed_time(e1)
        e2e = {"value": n_e2e * T / (e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": T * wl.H * 2, "d2h_bytes_per_step": T * wl.H * 2,
               "steps": n_e2e}

    if rank != 0:
        return
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        hbm_peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        hbm_peak, peak_src = 6800.0, "fallback"
    achieved = alg_bytes / (ms_per_step * 1e-3) / 1e9
    tokens_per_s = world * T * steps / (ms / 1e3)
    roofline = {"bound": "hbm",
                "kernel": ("decode_fused_kernel (the step's only launch)" if T <= 8
                           else "whole layer call (all launches of one step)"),
                "achieved": achieved, "peak": hbm_peak, "peak_source": peak_src,
                "unit": "GB/s", "frac": achieved / hbm_peak,
                "algorithmic_bytes_per_launch": alg_bytes,
                "traffic": NCU_TRAFFIC.get(args.workload)}
    if stage_ms and T >= 1024:
        # dense contraction: the up/gate grouped GEMM against the tensor peak
        # (fp16 operands; GB300's nominal fp16 and bf16 dense rates are equal,
        # so the measured sustained bf16 cuBLAS rate is the fp16 peak)
        routes = T * (wl.k + 1)
        ug_flop = routes * 4.0 * wl.H * wl.F
        try:
            tc_peak, tc_src = float(peaks["bf16_tflops_sustained"]), "measured (sustained bf16 = fp16)"
        except (KeyError, ValueError):
            tc_peak, tc_src = 1700.0, "fallback"
        ug_tflops = ug_flop / (stage_ms["up/gate"] * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": "grouped_gemm_tc<up/gate>",
                    "achieved": ug_tflops, "peak": tc_peak, "peak_source": tc_src,
                    "unit": "TFLOP/s", "frac": ug_tflops / tc_peak,
                    "algorithmic_flops_per_launch": ug_flop,
                    "launch_ms": stage_ms["up/gate"], "traffic": NCU_TRAFFIC.get(args.workload)}
    line = {
        "metric": METRIC,
        "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in/out, IQ4_NL weights, fp32 accumulate",
        "data": "synthetic (seeded; random IQ4_NL weights of the workload's layer shapes)",
        "config": cfg,
        "us_per_layer": ms_per_step * 1e3,
        "expert_weight_gbs": expert_bytes / (ms_per_step * 1e-3) / 1e9,
        "expert_weight_frac_of_hbm_peak": expert_bytes / (ms_per_step * 1e-3) / 1e9 / hbm_peak,
        "roofline": roofline,
        "stage_ms": stage_ms,
        "step_ms_percentiles": replay_percentiles(start, marks, G),
        "gpu_launches": gpu_launches,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def run_trunk(args, rank, world, local_rank):
    """A step is T tokens through the whole trunk: per layer a residual-add +
    RMSNorm launch and the layer's route + forward launches."""
    import numpy as np
    import torch
    import quantized_moe_expert_sigmoid_gb300 as moe
    from quantized_moe_expert_sigmoid_gb300 import build as moe_build, synth
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(moe_build.LIB):
        moe_build.build()
    if world > 1:
        torch.distributed.barrier()
    wl = synth.WORKLOADS[args.workload]
    T = wl.T
    NL, NX, G, cfg = bench_config(args, wl, world)
    layers, routers = [], []
    for l in range(NL):
        ew = synth.expert_weights_torch(1000 * rank + 7, l, wl.E, wl.H, wl.F, device=dev)
        layers.append(moe.MoeLayer(wl.H, wl.E, wl.k, wl.F, 1, wl.scale, T, up=ew.up, gate=ew.gate,
                                   down=ew.down, sh_up=ew.sh_up, sh_gate=ew.sh_gate,
                                   sh_down=ew.sh_down))
        del ew
        routers.append(torch.from_numpy(synth.router_weights(7, l, wl.E, wl.H, wl.router_sigma)).to(dev))
    torch.cuda.empty_cache()
    trunk = moe.MoeTrunk(layers, routers, T)
    xs_host = [synth.activations(100 + rank, "trunk", T, wl.H, np.full(T, i)) for i in range(NX)]
    xs = [torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16) for a in xs_host]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for j in range(max(3, args.warmup)):
            trunk.forward(xs[j % NX])
    stream.synchronize()
    trunk.check()

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(n):
                trunk.forward(xs[j % NX])
        return g

    reps, rem = divmod(args.steps, G)
    launches0 = moe.moe_launch_count()
    g_main = capture(G) if reps else None
    launches_per_graph = moe.moe_launch_count() - launches0
    launches0 = moe.moe_launch_count()
    g_rem = capture(rem) if rem else None
    launches_rem = moe.moe_launch_count() - launches0
    with torch.cuda.stream(stream):
        for g in (g_main, g_rem):
            if g:
                g.replay()
    stream.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    with Clocks(local_rank) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(reps):
                g_main.replay()
                marks[i].record(stream)
            if g_rem:
                g_rem.replay()
            stop.record(stream)
        stop.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = start.elapsed_time(stop)
    trunk.check()
    t_ms = torch.tensor([ms], device=dev)
    if world > 1:
        torch.distributed.all_reduce(t_ms, op=torch.distributed.ReduceOp.MAX)
    ms = float(t_ms.item())
    steps = reps * G + rem
    ms_per_step = ms / steps
    # bytes of the last step: every layer's selected experts + shared, routers, activations
    distinct = [len(set(trunk.ids[l][:T].flatten().tolist())) for l in range(NL)]
    expert_bytes = sum(d + 1 for d in distinct) * expert_bytes_of(wl)
    alg_bytes = expert_bytes + NL * (wl.E * wl.H * 4 + T * wl.H * (2 + 4 + 4 + 4 + 2))

    e2e = None
    if rank == 0:
        n_e2e = max(1, min(args.e2e_steps, args.steps, 200))
        xh = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory() for a in xs_host]
        rh = torch.empty((T, wl.H), dtype=torch.float32).pin_memory()
        xd = torch.empty((T, wl.H), dtype=torch.bfloat16, device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for j in range(4):
                xd.copy_(xh[j % NX], non_blocking=True)
                rh.copy_(trunk.forward(xd), non_blocking=True)
            stream.synchronize()
            e0.record(stream)
            for j in range(n_e2e):
                xd.copy_(xh[j % NX], non_blocking=True)
                rh.copy_(trunk.forward(xd), non_blocking=True)
            e1.record(stream)
        e1.synchronize()
        e2e = {"value": n_e2e * T / (e0.elapsed_time(e1) / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": T * wl.H * 2, "d2h_bytes_per_step": T * wl.H * 4,
               "steps": n_e2e}
    if rank != 0:
        return
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        hbm_peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        hbm_peak, peak_src = 6800.0, "fallback"
    achieved = alg_bytes / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": world * T * steps / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp32 residual, IQ4_NL weights, fp32 accumulate",
        "data": "synthetic (seeded; random IQ4_NL weights of the Xing4 trunk shapes)",
        "config": cfg,
        "us_per_layer": ms_per_step * 1e3 / NL,
        "expert_weight_gbs": expert_bytes / (ms_per_step * 1e-3) / 1e9,
        "expert_weight_frac_of_hbm_peak": expert_bytes / (ms_per_step * 1e-3) / 1e9 / hbm_peak,
        "step_ms_percentiles": replay_percentiles(start, marks, G),
        "roofline": {"bound": "hbm", "kernel": f"whole trunk step ({NL} layers, all launches)",
                     "achieved": achieved, "peak": hbm_peak, "peak_source": peak_src,
                     "unit": "GB/s", "frac": achieved / hbm_peak,
                     "algorithmic_bytes_per_launch": alg_bytes, "traffic": None},
        "gpu_launches": reps * launches_per_graph + launches_rem,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        if args.workload.startswith("trunk"):
            run_trunk(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
