"""Benchmark of the routed IQ4_NL MoE layer on GB300 (one JSON line on rank 0).

A step is one call of the whole layer (router logits, sigmoid top-k and
weights, per-expert histogram/scan/permutation, gather, dequantising
up/gate + SwiGLU, down projection, weighted combine with the shared expert)
over one batch of synthetic tokens.  Headline workload: the Xing4-shaped
layer at decode batch 1 (H 3584, 64 experts top-4 + 1 shared, F 1024, bf16
x).  The default run (one GPU) then measures the other configurations of the
same layer the same way and reports them under "workloads": the tiny layer,
batched decode of 64 tokens, the 4,096-token Zipf-skewed prefill, and the
38-layer trunk at 1 and 16 tokens.

L2: one layer's working set (~32 MB at batch 1) fits the 129 MB L2, so
steps rotate over NL resident layers with distinct weights (16 by default:
6.5 GB) and 64 distinct inputs; the data touched in one rotation (16 x 31.9
MB) is about 4x the L2, so each step's weights come from HBM.  Batches of 64
and more tokens touch ~400 MB per call and rotate over 2 layers; the trunk
holds its 38 layers (15.3 GB).

Steps run as CUDA-graph replays (G steps per graph) so that the GPU, not the
Python launch loop, sets the pace; the graph holds exactly the launches of G
layer calls, and the timed region replays it until exactly --steps steps
have run.  The spread of the step time (p10 / median / p90) comes from a
further >= 10 replays of the same graph, each timed on its own.  `e2e` times
the same calls eagerly, one moe_layer_forward_routed_host call per step: the
input taken from pinned host memory, the layer, and the output written back
to pinned host memory, all inside the timed region.  Up to 16 tokens the
decode kernels bring x across the host link themselves and store out through
it; above that the library enqueues copies.  The byte counts are those of x
and out either way.

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

# configurations measured beside the decode-1 headline in the default run
EXTRA_WORKLOADS = ("tiny", "decode64", "prefill4096", "trunk38_t1", "trunk38_t16")


def expert_bytes_of(wl):
    """IQ4_NL bytes of one expert: up, gate and down, 18 bytes per 32 weights
    (6,193,152 B for the Xing4 layer)."""
    return 3 * wl.F * (wl.H // 32) * 18


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode1",
                   choices=["tiny", "decode1", "decode8", "decode64", "prefill4096", "trunk38_t1", "trunk38_t16",
                            "k2h_decode1", "k2h_decode64", "k2h_prefill1024"])
    p.add_argument("--layers", type=int, default=16, help="resident layers the steps rotate over")
    p.add_argument("--graph-steps", type=int, default=32)
    p.add_argument("--e2e-steps", type=int, default=2000)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true",
                   help="measure the headline workload only (no 'workloads' section)")
    return p.parse_args()


METRIC = "MoE-layer tokens/s (expert-weight HBM GB/s as fraction of GB300 peak)"

# DRAM bytes (read + write) per launch of each workload's dominant kernel,
# from the ncu captures summarised in profiles/ (None when the kernel changed
# after its capture).
NCU_TRAFFIC = {
    "decode1": 32_084_480,        # decode_unit_kernel<14,2>, ncu dram read + write per launch
    "decode8": None,              # decode_batch_kernel<14,2,false>: changed after its capture (counter layout)
    "prefill4096": 457_219_328,   # grouped_gemm_tc<up/gate>, ncu dram read + write per launch
}


def load_peaks():
    """Roofline denominators: MEASURED_PEAKS.json, else the fallback figures."""
    try:
        pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return {"hbm": float(pk["hbm_gbs"]), "hbm_src": "measured",
                "bf16": float(pk["bf16_tflops"]), "bf16_src": "measured burst",
                "bf16_sus": float(pk["bf16_tflops_sustained"]), "bf16_sus_src": "measured sustained"}
    except (OSError, KeyError, ValueError):
        return {"hbm": 6800.0, "hbm_src": "fallback", "bf16": 1900.0, "bf16_src": "fallback burst",
                "bf16_sus": 1700.0, "bf16_sus_src": "fallback sustained"}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def bench_config(args, wl, world, steps):
    """(resident layers, distinct inputs, steps per graph, config dict)."""
    T = wl.T
    if wl.n_layers > 1:
        G = max(1, min(args.graph_steps, steps, 8))
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
    G = max(1, min(args.graph_steps, steps))
    return NL, NX, G, {
        "workload": wl.name, "tokens_per_step": T, "hidden": wl.H, "experts": wl.E,
        "top_k": wl.k, "expert_ffn": wl.F, "shared_experts": 1, "routed_scaling": wl.scale,
        "parallelism": f"replicas x{world}",
        "l2": f"rotating over {NL} resident layers and {NX} inputs (inputs larger than L2)",
        "graph_steps": G}


def algorithmic_bytes(wl, T, distinct_experts):
    """HBM bytes one call must move at least: the selected experts' and the
    shared expert's IQ4_NL weights, the fp32 router, x in and out (bf16)."""
    return (distinct_experts + 1) * expert_bytes_of(wl) + wl.E * wl.H * 4 + 2 * T * wl.H * 2


def layer_flops(wl, T):
    """Dense-equivalent flops of one call: 6 H F per route (gate, up, down
    multiply-adds) for the k routed and the shared expert, plus the fp32
    router's 2 T E H."""
    return T * (wl.k + 1) * 6.0 * wl.H * wl.F + 2.0 * T * wl.E * wl.H


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
        x = oracle.to_f64(synth.activations(0, "bench", 1, wl.H, np.array([done]), wl.x_dtype), wl.x_dtype)
        b = None if bias is None else bias[done % wl.T][None, :]
        oracle.moe_layer(x, wr, ew, wl.k, wl.scale, b)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    cores = host_cores()
    if wl.n_layers > 1:  # a token crosses every layer of the trunk (plus an RMSNorm each)
        return {"value": done / el / wl.n_layers, "unit": "tokens/s", "cores": 1, "host_cores": cores,
                "kind": "oracle",
                "sample": f"{done} single-token calls of one layer of the {wl_name} trunk "
                          f"({el:.1f} s, fp64, 1 thread of {cores}), scaled by its {wl.n_layers} layers"}
    return {"value": done / el, "unit": "tokens/s", "cores": 1, "host_cores": cores, "kind": "oracle",
            "sample": f"{done} single-token layer calls of the {wl_name} workload "
                      f"({el:.1f} s, fp64, 1 thread of {cores})"}


def run_reference(args, rank, world):
    from quantized_moe_expert_sigmoid_gb300 import synth
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    budget = 90.0
    r = cpu_baseline(args.workload, min(budget, 3.0 + 0.2 * (args.steps + args.warmup)))
    _, _, _, cfg = bench_config(args, wl, world, args.steps)
    line = {"impl": "reference", "metric": METRIC, "value": r["value"],
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "ms_per_step": 1000.0 * wl.T / r["value"],
            "cpu_baseline": r,
            "e2e": {"value": r["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def timed_graph_steps(torch, moe, stream, step, steps, G, local_rank, world):
    """Capture G steps in a graph (and the remainder in a second), replay
    them so that exactly `steps` steps run in the timed region, bracketed by
    a barrier and device synchronisations; then time >= 10 further replays
    one by one for the spread.  Returns (ms, launches in the timed region,
    clocks summary, percentiles)."""
    reps, rem = divmod(steps, G)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(n):
                step(j, j)
        return g

    l0 = moe.moe_launch_count()
    g_main = capture(G) if reps else None
    per_graph = moe.moe_launch_count() - l0
    l0 = moe.moe_launch_count()
    g_rem = capture(rem) if rem else None
    per_rem = moe.moe_launch_count() - l0
    with torch.cuda.stream(stream):
        for g in (g_main, g_rem):
            if g:
                g.replay()
    stream.synchronize()

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(local_rank) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(reps):
                g_main.replay()
            if g_rem:
                g_rem.replay()
            stop.record(stream)
        stop.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = start.elapsed_time(stop)

    # spread: replays of the main graph, each timed on its own (outside the
    # timed region above)
    g_spread, n_steps = (g_main, G) if g_main else (g_rem, rem)
    per_replay_ms = ms / max(1, steps) * n_steps
    n_rep = int(max(10, min(200, 2000.0 / max(per_replay_ms, 1e-3))))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(n_rep):
            g_spread.replay()
            ev[i + 1].record(stream)
    ev[-1].synchronize()
    ts = sorted(ev[i].elapsed_time(ev[i + 1]) / n_steps for i in range(n_rep))
    pick = lambda q: ts[min(len(ts) - 1, int(q * (len(ts) - 1) + 0.5))]
    pct = {"p10": pick(0.1), "median": pick(0.5), "p90": pick(0.9), "replays": n_rep,
           "steps_per_replay": n_steps, "where": "replays after the timed region, each timed on its own"}
    del g_main, g_rem, g_spread
    return ms, reps * per_graph + (per_rem if rem else 0), clk.summary(), pct


def measure_layer(args, name, steps, warmup, world, rank, local_rank, dev, cpu_seconds, headline):
    """One single-layer workload: bench line fields (value, ms, roofline, ...)."""
    import numpy as np
    import torch
    import quantized_moe_expert_sigmoid_gb300 as moe
    from quantized_moe_expert_sigmoid_gb300 import synth

    wl = synth.WORKLOADS[name]
    T = wl.T
    NL, NX, G, cfg = bench_config(args, wl, world, steps)
    pk = load_peaks()

    layers, routers = [], []
    for l in range(NL):
        ew = synth.expert_weights_torch(1000 * rank + 7, l, wl.E, wl.H, wl.F, device=dev)
        layers.append(moe.MoeLayer(wl.H, wl.E, wl.k, wl.F, 1, wl.scale, T, up=ew.up, gate=ew.gate,
                                   down=ew.down, sh_up=ew.sh_up, sh_gate=ew.sh_gate,
                                   sh_down=ew.sh_down, flags=moe.MOE_FLAG_HOST_IO))
        del ew
        routers.append(torch.from_numpy(synth.router_weights(7, l, wl.E, wl.H, wl.router_sigma)).to(dev))
    torch.cuda.empty_cache()
    xs_host = [synth.activations(100 + rank, "bench", T, wl.H, np.full(T, i), wl.x_dtype) for i in range(NX)]
    xdt = torch.bfloat16 if wl.x_dtype == "bf16" else torch.float32

    def to_x(a, device=None):
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if wl.x_dtype == "bf16" else torch.from_numpy(a)
        return t.to(device) if device is not None else t

    xs = [to_x(a, dev) for a in xs_host]
    bias = torch.from_numpy(synth.zipf_logit_bias(7, T, wl.E)).to(dev) if wl.zipf else None
    outs = [torch.empty((T, wl.H), dtype=xdt, device=dev) for _ in range(G)]
    ids = [torch.empty((T, wl.k), dtype=torch.int32, device=dev) for _ in range(G)]
    wts = [torch.empty((T, wl.k), dtype=torch.float32, device=dev) for _ in range(G)]

    def step(j, slot):
        L = layers[j % NL]
        moe.moe_layer_forward_routed(L.handle, xs[j % NX], routers[j % NL], ids[slot], wts[slot],
                                     outs[slot], bias)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for j in range(max(3, warmup)):
            step(j, j % G)
    stream.synchronize()
    for L in layers:
        L.check()

    # the batched path has several kernels per call: its stages are timed
    # with CUDA events recorded inside the graph (event-record nodes that
    # every replay refreshes), so the dominant kernel's own duration is
    # measured in the timed region
    staged = T > 8
    if staged:
        for L in layers:
            moe.moe_layer_enable_timing(L.handle, G)
    ms, gpu_launches, clocks, pct = timed_graph_steps(torch, moe, stream, step, steps, G, local_rank, world)
    for L in layers:
        L.check()
    t_ms = torch.tensor([ms], device=dev)
    if world > 1:
        torch.distributed.all_reduce(t_ms, op=torch.distributed.ReduceOp.MAX)
    ms = float(t_ms.item())
    stage_ms = None
    if staged:  # per-stage means over the calls of the last replay
        rows = [r for L in layers for r in moe.moe_layer_stage_times(L.handle, G)]
        stage_ms = {nm: statistics.fmean(r[i] for r in rows) for i, nm in enumerate(moe.STAGES)}
        for L in layers:  # the events stay bound to the graphs: fresh ones before eager calls
            moe.moe_layer_enable_timing(L.handle, 0)
    ms_per_step = ms / steps

    # distinct experts selected per step (for the byte count)
    distinct = [len(set(ids[s].flatten().tolist())) for s in range(min(G, steps))]
    mean_distinct = sum(distinct) / len(distinct)
    alg_bytes = algorithmic_bytes(wl, T, mean_distinct)
    expert_bytes = (mean_distinct + 1) * expert_bytes_of(wl)

    # end to end through the public API with host buffers
    e2e = None
    if rank == 0:
        n_e2e = max(1, min(args.e2e_steps, steps))
        xh = [to_x(a).pin_memory() for a in xs_host]
        oh = torch.empty((T, wl.H), dtype=xdt).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for j in range(8):  # one C-ABI call per step: copy x in, run the layer, copy out back
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
        nbytes = T * wl.H * (2 if wl.x_dtype == "bf16" else 4)
        e2e = {"value": world * n_e2e * T / (e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "steps": n_e2e,
               "us_per_step": 1e3 * e_ms / n_e2e}
    for L in layers:
        L.check()
        L.close()
    del layers, routers, xs, outs, ids, wts
    torch.cuda.empty_cache()

    achieved = alg_bytes / (ms_per_step * 1e-3) / 1e9
    if wl.n_layers > 1:
        kname = "whole trunk step (every layer's calls and the residual RMSNorm launches)"
    elif T == 1:
        kname = "decode_unit_kernel (the step's only launch)"
    elif T <= 16 and wl.H in (3584, 2560):
        kname = "decode_batch_kernel (the step's only launch)"
    elif T <= 8:
        kname = "decode_fused_kernel (the step's only launch)"
    else:
        kname = "whole layer call (all launches of one step)"
    roofline = {"bound": "hbm",
                "kernel": kname,
                "achieved": achieved, "peak": pk["hbm"], "peak_source": pk["hbm_src"],
                "unit": "GB/s", "frac": achieved / pk["hbm"],
                "algorithmic_bytes_per_launch": alg_bytes,
                "traffic": NCU_TRAFFIC.get(name) if T <= 8 and wl.n_layers == 1 else None}
    out = {"value": world * T * steps / (ms / 1e3), "unit": "tokens/s", "steps": steps,
           "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1e3, "config": cfg,
           "expert_weight_gbs": expert_bytes / (ms_per_step * 1e-3) / 1e9,
           "expert_weight_frac_of_hbm_peak": expert_bytes / (ms_per_step * 1e-3) / 1e9 / pk["hbm"],
           "mean_distinct_experts": mean_distinct}
    if stage_ms and T >= 1024:
        # dense contraction: the up/gate grouped GEMM (a sub-millisecond
        # kernel, so the burst bf16 peak; fp16 operands, and GB300's fp16 and
        # bf16 dense rates are equal) against the tensor roofline, and the
        # whole call's dense-equivalent flops beside it
        routes = T * (wl.k + 1)
        ug_flop = routes * 4.0 * wl.H * wl.F
        ug_tflops = ug_flop / (stage_ms["up/gate"] * 1e-3) / 1e12
        out["hbm_roofline_of_call"] = roofline
        roofline = {"bound": "tensor", "kernel": "grouped_gemm_tc<up/gate>",
                    "achieved": ug_tflops, "peak": pk["bf16"], "peak_source": pk["bf16_src"] + " (fp16 = bf16 rate)",
                    "unit": "TFLOP/s", "frac": ug_tflops / pk["bf16"],
                    "algorithmic_flops_per_launch": ug_flop,
                    "launch_ms": stage_ms["up/gate"], "traffic": NCU_TRAFFIC.get(name)}
        call_tflops = layer_flops(wl, T) / (ms_per_step * 1e-3) / 1e12
        out["whole_layer_tensor"] = {"achieved": call_tflops, "peak": pk["bf16"], "unit": "TFLOP/s",
                                     "frac": call_tflops / pk["bf16"],
                                     "flops_per_call": layer_flops(wl, T),
                                     "peak_source": pk["bf16_src"]}
    out.update({"roofline": roofline, "stage_ms": stage_ms, "step_ms_percentiles": pct,
                "gpu_launches": gpu_launches, "clocks": clocks, "e2e": e2e})
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(name, cpu_seconds)
    return out


def measure_trunk(args, name, steps, warmup, world, rank, local_rank, dev, cpu_seconds, headline):
    """A step is T tokens through the whole trunk: per layer a residual-add +
    RMSNorm launch and the layer's route + forward launches."""
    import numpy as np
    import torch
    import quantized_moe_expert_sigmoid_gb300 as moe
    from quantized_moe_expert_sigmoid_gb300 import synth
    wl = synth.WORKLOADS[name]
    T = wl.T
    NL, NX, G, cfg = bench_config(args, wl, world, steps)
    pk = load_peaks()
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
        for j in range(max(3, warmup)):
            trunk.forward(xs[j % NX])
    stream.synchronize()
    trunk.check()

    def step(j, slot):
        trunk.forward(xs[j % NX])

    ms, gpu_launches, clocks, pct = timed_graph_steps(torch, moe, stream, step, steps, G, local_rank, world)
    trunk.check()
    t_ms = torch.tensor([ms], device=dev)
    if world > 1:
        torch.distributed.all_reduce(t_ms, op=torch.distributed.ReduceOp.MAX)
    ms = float(t_ms.item())
    ms_per_step = ms / steps
    # bytes of the last step: every layer's selected experts + shared, routers, activations
    distinct = [len(set(trunk.ids[l][:T].flatten().tolist())) for l in range(NL)]
    expert_bytes = sum(d + 1 for d in distinct) * expert_bytes_of(wl)
    alg_bytes = expert_bytes + NL * (wl.E * wl.H * 4 + T * wl.H * (2 + 4 + 4 + 4 + 2))

    e2e = None
    if rank == 0:
        n_e2e = max(1, min(args.e2e_steps, steps, 200))
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
        e2e = {"value": world * n_e2e * T / (e0.elapsed_time(e1) / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": T * wl.H * 2, "d2h_bytes_per_step": T * wl.H * 4,
               "steps": n_e2e}
    for L in layers:
        L.close()
    del trunk, layers, routers, xs
    torch.cuda.empty_cache()
    achieved = alg_bytes / (ms_per_step * 1e-3) / 1e9
    out = {"value": world * T * steps / (ms / 1e3), "unit": "tokens/s", "steps": steps,
           "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1e3 / NL, "config": cfg,
           "expert_weight_gbs": expert_bytes / (ms_per_step * 1e-3) / 1e9,
           "expert_weight_frac_of_hbm_peak": expert_bytes / (ms_per_step * 1e-3) / 1e9 / pk["hbm"],
           "expert_bytes_per_token": expert_bytes / T,
           "step_ms_percentiles": pct,
           "roofline": {"bound": "hbm", "kernel": f"whole trunk step ({NL} layers, all launches)",
                        "achieved": achieved, "peak": pk["hbm"], "peak_source": pk["hbm_src"],
                        "unit": "GB/s", "frac": achieved / pk["hbm"],
                        "algorithmic_bytes_per_launch": alg_bytes, "traffic": None},
           "gpu_launches": gpu_launches, "clocks": clocks, "e2e": e2e}
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(name, cpu_seconds)
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    from quantized_moe_expert_sigmoid_gb300 import build as moe_build, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(moe_build.LIB):
        moe_build.build()
    if world > 1:
        torch.distributed.barrier()

    def measure(name, steps, warmup, cpu_s, headline):
        f = measure_trunk if synth.WORKLOADS[name].n_layers > 1 else measure_layer
        return f(args, name, steps, warmup, world, rank, local_rank, dev, cpu_s, headline)

    head = measure(args.workload, args.steps, args.warmup, args.cpu_seconds, True)
    extra = {}
    if world == 1 and not args.no_extra and args.workload == "decode1":
        for name in EXTRA_WORKLOADS:
            wl = synth.WORKLOADS[name]
            # bounded: at least 20 steps, about a second of timed work each
            n = max(20, min(args.steps, 200 if wl.T <= 64 and wl.n_layers == 1 else 40))
            extra[name] = measure(name, n, max(3, min(args.warmup, 10)), min(args.cpu_seconds, 4.0), False)
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in/out, IQ4_NL weights, fp32 accumulate",
        "data": "synthetic (seeded; random IQ4_NL weights of the workload's layer shapes)",
        "config": head["config"],
    }
    for k, v in head.items():
        if k not in ("value", "unit", "steps", "ms_per_step", "config"):
            line[k] = v
    if extra:
        line["workloads"] = extra
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
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
