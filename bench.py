#!/usr/bin/env python
"""Benchmark of the GB300 4-bit MoE layer: MoE-layer tokens/s and fraction of roofline.

Headline workload: decode, batch 1 (T = 1, d = 2048, E = 256, top-8, SwiGLU width 512, shared
expert with sigmoid gate, 4-bit affine group-64 weights).  One step = one decode token through 40
MoE layers, each with its own seeded weight set (40 x 455 MB = 18.2 GB resident in HBM, cycled, so
no layer's experts are in L2 when it runs) and its own precomputed input row.  `value` counts
MoE-layer tokens per second (40 per step per GPU).  The line also carries, under `prefill`,
one layer call at T = 512 and at T = 4096 (Zipf-skewed routing) and the 40-layer stack at
T = 2048 (pre-norm block + layer per layer), the two layer calls again with bf16 tensor-core
operands (`operands`: "bf16"), and a hot-L2 single-layer decode figure.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extras]

Under torchrun (N > 1) every rank runs the same workload on its own GPU (independent replicas; the
layer has no cross-GPU exchange) and rank 0 prints one JSON line with the whole-job rate.
`--impl reference` times the CPU oracle (float64 numpy) on the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
_T0 = time.perf_counter()


def log(msg):
    print(f"[bench {time.perf_counter() - _T0:7.1f}s] {msg}", file=sys.stderr, flush=True)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s (decode T=1, prefill T=512/4096); % of HBM/tensor roofline"
LAYERS = 40
NI = 64   # distinct input rows per layer for decode
# dram__bytes_read.sum + dram__bytes_write.sum of one decode layer call (its decode_layer_kernel and
# decode_reduce_kernel launches) at the decode shape, from one ncu capture of
# `bench.py --profile decode`; None whenever those kernels have changed since the capture.
DECODE_NCU_TRAFFIC = 16300672


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extras", action="store_true", help="skip the prefill T=512 / T=4096 sub-measurements")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--profile", choices=["decode", "prefill", "skewed", "stack", "attention", "scan"], default=None,
                   help="small eager run of one workload for ncu captures (prints a short summary only)")
    p.add_argument("--profile-sets", type=int, default=4, help="weight sets cycled in --profile mode")
    p.add_argument("--profile-operands", choices=["fp16", "bf16"], default="fp16",
                   help="tensor-core operand type of the grouped-GEMM path in --profile mode")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------------------ algorithmic work

def qmat_bytes(R, C):
    return R * C // 2 + 2 * R * (C // 64) * 2


def expert_bytes(wl):
    return 2 * qmat_bytes(wl.F, wl.d) + qmat_bytes(wl.d, wl.F)


def layer_bytes(wl, T, touched_experts):
    """Weights of the experts the tokens actually use (+ shared) + x, logits, w_sg, y."""
    w = (touched_experts + (1 if wl.F_shared else 0)) * expert_bytes(wl)
    io = T * wl.d * 2 + T * wl.E * 4 + wl.d * 2 + T * wl.d * 4
    return w + io


def layer_flops(wl, T):
    return 6 * wl.d * wl.F * (T * wl.k + (T if wl.F_shared else 0))


# ------------------------------------------------------------------------------ clocks

class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return out
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        out.update({"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                    "reasons": reasons, "samples": len(rows)})
        return out


# ------------------------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------ ours

def make_layers(wl, device, n):
    import bit_quantized_expert_gb300 as moe
    layers = []
    for l in range(n):
        t = synth.torch_make_layer(wl, seed=l, device=device)
        layers.append(moe.Layer(t["routed"], t["shared"], t["w_sg"], wl.d, wl.E, wl.k, wl.F))
    return layers


def on_stream(stream):
    """Context that makes `stream` current after it waits for the work already queued on the
    default stream.  Inputs, weights and workspace clears are made there, and a side stream does
    not wait for the default stream by itself."""
    import torch
    stream.wait_stream(torch.cuda.default_stream(stream.device))
    return torch.cuda.stream(stream)


def capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def timed_graph_steps(graph_of_g, g_steps, graph_of_1, steps, stream):
    """Replay graphs so that exactly `steps` steps run; returns elapsed ms (CUDA events on `stream`)."""
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps, rest = divmod(steps, g_steps)
    with on_stream(stream):
        start.record(stream)
        for _ in range(reps):
            graph_of_g.replay()
        for _ in range(rest):
            graph_of_1.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


def decode_bench(args, world, rank, local, device, pk):
    import torch

    import bit_quantized_expert_gb300 as moe
    wl = synth.DECODE
    log("decode: generating 40 weight sets on the device")
    layers = make_layers(wl, device, LAYERS)
    ins = [synth.torch_make_inputs(wl, seed=1000 + l, device=device, T=NI) for l in range(LAYERS)]
    y = torch.empty((LAYERS, NI, wl.d), dtype=torch.float32, device=device)
    dm = layers[0].dims(1)
    ws = moe.alloc_workspace(dm, device)
    stream = torch.cuda.Stream(device=device)

    def step(s):
        i = s % NI
        for l in range(LAYERS):
            layers[l].forward(ins[l]["x"][i:i + 1], ins[l]["logits"][i:i + 1], y[l, i:i + 1], ws)

    with on_stream(stream):
        for s in range(args.warmup):
            step(s)
    stream.synchronize()
    G = 25
    log("decode: warm-up done; capturing graphs")
    g_many = capture(lambda: [step(s) for s in range(G)], stream)
    g_one = capture(lambda: step(0), stream)
    with on_stream(stream):
        g_many.replay()
    stream.synchronize()
    if moe.read_error_flags(ws) != 0:
        raise RuntimeError("device error flags set during warm-up")

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = Clocks(vis.split(",")[local] if vis else local)
    torch.cuda.synchronize()
    barrier(world)
    log(f"decode: timing {args.steps} steps")
    clocks.start()
    ms = timed_graph_steps(g_many, G, g_one, args.steps, stream)
    ck = clocks.stop()
    log(f"decode: {ms / args.steps * 1e3:.2f} us per step")
    torch.cuda.synchronize()
    barrier(world)
    flags = moe.read_error_flags(ws)
    ms_max = max_over_ranks(ms, world, device)

    # Expert touches per layer call: k routed (distinct) + shared; algorithmic bytes of one call.
    per_call = layer_bytes(wl, 1, wl.k)
    per_step_bytes = LAYERS * per_call
    step_s = ms_max / 1e3 / args.steps
    tokens = LAYERS * args.steps * world
    res = {
        "value": tokens / (ms_max / 1e3), "ms_per_step": ms_max / args.steps, "clocks": ck, "flags": flags,
        "roofline": {"kernel": "decode_layer_kernel + decode_reduce_kernel (the two launches of a layer call)",
                     "bound": "hbm", "achieved": per_step_bytes / step_s / 1e9, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": per_step_bytes / step_s / 1e9 / pk["hbm_gbs"],
                     "traffic": DECODE_NCU_TRAFFIC,
                     "algorithmic_bytes_per_launch": per_call, "peak_source": pk["source"]},
        "gpu_launches": 2 * LAYERS * args.steps,   # decode_layer_kernel and decode_reduce_kernel per layer call
    }

    # Hot-L2 single-layer figure (labelled as such, not the headline): one weight set, replayed,
    # so its 16 MB of weights stay in L2.
    def hot_step(s):
        i = s % NI
        layers[0].forward(ins[0]["x"][i:i + 1], ins[0]["logits"][i:i + 1], y[0, i:i + 1], ws)

    with on_stream(stream):
        for s in range(3):
            hot_step(s)
    g_hot = capture(lambda: [hot_step(s) for s in range(LAYERS)], stream)
    with on_stream(stream):
        g_hot.replay()
    stream.synchronize()
    hot_calls = LAYERS * max(1, args.steps // 4)
    hot_ms = timed_graph_steps(g_hot, LAYERS, g_hot, hot_calls - hot_calls % LAYERS, stream)
    res["hot_l2"] = {"us_per_layer": hot_ms * 1e3 / (hot_calls - hot_calls % LAYERS),
                     "note": "one weight set replayed (weights L2-resident); not the headline"}
    log(f"decode hot-L2: {res['hot_l2']['us_per_layer']:.2f} us per layer")

    # Bandwidth ceiling of the decode access pattern: the loads-only replica of the decode launch
    # (same grid, clusters, copies and programmatic launch; experts given, no arithmetic) over the
    # same 40 weight sets and the same routing as the timed steps.
    idx = []
    for l in range(LAYERS):
        r = moe.alloc_routing(layers[l].dims(NI), 112, device)
        ws_r = moe.alloc_workspace(layers[l].dims(NI), device)
        moe.route(layers[l].dims(NI), ins[l]["logits"], r, ws_r)
        idx.append(r["idx"].clone())
        del r, ws_r
    torch.cuda.synchronize()

    def probe_step(s):
        i = s % NI
        for l in range(LAYERS):
            moe.decode_stream_probe(dm, idx[l][i], layers[l].routed, layers[l].shared, ws)

    with on_stream(stream):
        for s in range(3):
            probe_step(s)
    g_probe = capture(lambda: [probe_step(s) for s in range(G)], stream)
    with on_stream(stream):
        g_probe.replay()
    stream.synchronize()
    p_steps = max(G, args.steps // 2 // G * G)
    p_ms = timed_graph_steps(g_probe, G, g_probe, p_steps, stream)
    p_us = p_ms * 1e3 / (p_steps * LAYERS)
    res["loads_only"] = {"us_per_layer": p_us, "GB_s": per_call / (p_us * 1e-6) / 1e9,
                         "frac": per_call / (p_us * 1e-6) / 1e9 / pk["hbm_gbs"],
                         "note": "loads-only replica of the decode launch (moe_decode_stream_probe): same grid, "
                                 "clusters, shared memory, weight copies and programmatic launch, experts given, "
                                 "no arithmetic; the bandwidth ceiling of this access pattern"}
    if moe.read_error_flags(ws) != 0:
        raise RuntimeError("device error flags set during the loads-only runs")
    log(f"decode loads-only: {p_us:.2f} us per layer ({res['loads_only']['GB_s']:.0f} GB/s)")

    # A few tokens per layer call (verify-batch shapes): up to eight run the decode kernel in one
    # launch.  CUDA graph over the 40 weight sets; context, not the headline.
    small = {}
    ys = torch.empty((4, wl.d), dtype=torch.float32, device=device)
    for T in (2, 3, 4):
        ws_s = moe.alloc_workspace(layers[0].dims(T), device)

        def small_step(s, T=T, ws_s=ws_s):
            i = (s * T) % (NI - T)
            for l in range(LAYERS):
                layers[l].forward(ins[l]["x"][i:i + T], ins[l]["logits"][i:i + T], ys[:T], ws_s)

        with on_stream(stream):
            small_step(0)
        g_s = capture(lambda: [small_step(s) for s in range(4)], stream)
        with on_stream(stream):
            g_s.replay()
        stream.synchronize()
        reps = max(1, args.steps // 40)
        ms_s = timed_graph_steps(g_s, 4, g_s, 4 * reps, stream)
        per_layer = ms_s * 1e3 / (4 * reps * LAYERS)
        small[f"T{T}"] = {"us_per_layer": per_layer, "tokens_per_s": T * 1e6 / per_layer}
        if moe.read_error_flags(ws_s) != 0:
            raise RuntimeError("device error flags set during the small-T runs")
    res["small_T"] = small
    log("decode small T: " + ", ".join(f"{k} {v['us_per_layer']:.1f} us/layer" for k, v in small.items()))

    # End to end through the C ABI with host buffers: one moe_layer_forward_host call per layer.
    # The buffers are pinned (mapped into the device's address space), so the decode kernel reads
    # x and logits from host memory and writes y there itself; the bytes still cross the CPU-GPU
    # link inside the timed region, without copy-engine transfers on the stream.
    xh = [ins[l]["x"].cpu().pin_memory() for l in range(LAYERS)]
    lh = [ins[l]["logits"].cpu().pin_memory() for l in range(LAYERS)]
    yh = torch.empty((LAYERS, NI, wl.d), dtype=torch.float32).pin_memory()
    ws_h = moe.alloc_workspace_host(layers[0].dims(1), device)

    sh = stream.cuda_stream
    xs = [[xh[l][i:i + 1] for i in range(NI)] for l in range(LAYERS)]   # host views, made once
    ls = [[lh[l][i:i + 1] for i in range(NI)] for l in range(LAYERS)]
    ys = [[yh[l, i:i + 1] for i in range(NI)] for l in range(LAYERS)]

    # The step's inputs are in host memory before the step is queued: MOE_OPT_HOST_INPUTS_READY.
    def e2e_step(s):
        i = s % NI
        for l in range(LAYERS):
            layers[l].forward_host(xs[l][i], ls[l][i], ys[l][i], ws_h, sh, inputs_ready=True)

    # The same through staged copies: x and logits copied to device buffers, the device-pointer
    # layer call, y copied back (three copy-engine transfers per layer call on the stream).
    xd = torch.empty((1, wl.d), dtype=torch.int16, device=device)
    ld = torch.empty((1, wl.E), dtype=torch.float32, device=device)
    yd = torch.empty((1, wl.d), dtype=torch.float32, device=device)

    def staged_step(s):
        i = s % NI
        for l in range(LAYERS):
            xd.copy_(xs[l][i], non_blocking=True)
            ld.copy_(ls[l][i], non_blocking=True)
            layers[l].forward(xd, ld, yd, ws, stream=sh)
            ys[l][i].copy_(yd, non_blocking=True)

    n_e2e = max(1, min(args.steps, args.e2e_steps))

    def timed_host_steps(fn):
        with on_stream(stream):
            for s in range(2):
                fn(s)
            stream.synchronize()
            barrier(world)
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for s in range(n_e2e):
                fn(s)
            t1.record(stream)
        t1.synchronize()
        return max_over_ranks(t0.elapsed_time(t1), world, device)

    e2e_ms = timed_host_steps(e2e_step)
    staged_ms = timed_host_steps(staged_step)
    res["e2e"] = {"value": LAYERS * n_e2e * world / (e2e_ms / 1e3), "unit": "tokens/s",
                  "h2d_bytes_per_step": LAYERS * (wl.d * 2 + wl.E * 4), "d2h_bytes_per_step": LAYERS * wl.d * 4,
                  "steps": n_e2e,
                  "launch": "one moe_layer_forward_host_opts call per layer on pinned host buffers "
                            "(MOE_OPT_HOST_INPUTS_READY: inputs written by the host before the step): a "
                            "staging kernel reads x and logits from host memory, the decode kernel writes "
                            "y there"}
    res["e2e_staged"] = {"value": LAYERS * n_e2e * world / (staged_ms / 1e3), "unit": "tokens/s",
                         "launch": "per layer call: 2 H2D copies, moe_layer_forward on device buffers, "
                                   "1 D2H copy, all on one stream"}
    log(f"decode e2e: {res['e2e']['value']:.0f} tokens/s zero-copy, {res['e2e_staged']['value']:.0f} staged")
    if moe.read_error_flags(ws_h) != 0 or moe.read_error_flags(ws) != 0:
        raise RuntimeError("device error flags set during the end-to-end runs")
    del layers
    torch.cuda.empty_cache()
    return res


def prefill_bench(wl, steps, device, pk, operands="fp16"):
    """One step = one layer call over T tokens; 40 weight sets cycled; CUDA-graph replay.
    operands: the grouped GEMM's tensor-core operand type ("fp16", or "bf16" through
    moe_layer_forward_opts)."""
    import torch

    import bit_quantized_expert_gb300 as moe
    n_sets = 8 if wl.T >= 4096 else 16
    log(f"{wl.name} ({operands} operands): generating {n_sets} weight sets")
    layers = make_layers(wl, device, n_sets)
    ins = [synth.torch_make_inputs(wl, seed=1000 + l, device=device) for l in range(n_sets)]
    y = torch.empty((wl.T, wl.d), dtype=torch.float32, device=device)
    dm = layers[0].dims(wl.T)
    ws = moe.alloc_workspace(dm, device)
    routing = moe.alloc_routing(dm, 112, device)
    stream = torch.cuda.Stream(device=device)

    def step(s):
        l = s % n_sets
        layers[l].forward(ins[l]["x"], ins[l]["logits"], y, ws, operands=operands)

    with on_stream(stream):
        for s in range(3):
            step(s)
    stream.synchronize()
    g_many = capture(lambda: [step(s) for s in range(n_sets)], stream)
    g_one = capture(lambda: step(0), stream)
    with on_stream(stream):
        g_many.replay()
    stream.synchronize()
    steps = max(n_sets, steps // n_sets * n_sets)
    ms = timed_graph_steps(g_many, n_sets, g_one, steps, stream)
    log(f"{wl.name} ({operands} operands): {ms / steps * 1e3:.1f} us per step")
    flags = moe.read_error_flags(ws)
    # touched experts per weight set (from the routing of that set's inputs)
    touched = []
    for l in range(n_sets):
        with on_stream(stream):
            layers[l].forward(ins[l]["x"], ins[l]["logits"], y, ws, routing=routing, operands=operands)
        stream.synchronize()
        touched.append(int((routing["counts"] > 0).sum().item()))
    step_s = ms / 1e3 / steps
    bytes_avg = sum(layer_bytes(wl, wl.T, t) for t in touched) / n_sets
    flops = layer_flops(wl, wl.T)
    out = {"workload": wl.name, "operands": operands, "value": wl.T / step_s, "unit": "tokens/s",
           "ms_per_step": ms / steps,
           "steps": steps, "weight_sets": n_sets, "flags": flags,
           "hbm": {"achieved": bytes_avg / step_s / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                   "frac": bytes_avg / step_s / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": bytes_avg},
           "tensor": {"achieved": flops / step_s / 1e12, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                      "frac": flops / step_s / 1e12 / pk["bf16_tflops"], "algorithmic_flops": flops,
                      "note": f"{operands} operands; peak is the measured bf16 dense rate (fp16 and bf16 share "
                              "the nominal rate)"},
           # top-k, chunk histogram, chunk scan (with the GEMM walk order), chunk scatter, x permute,
           # gate/up GEMM, down GEMM, combine
           "gpu_launches_per_step": 8}
    del layers
    torch.cuda.empty_cache()
    return out


def stack_bench(wl, steps, device, pk):
    """One step = the token batch through 40 layers, each a pre-norm block (residual add, RMSNorm,
    router GEMM: moe_rmsnorm_router) and the MoE layer; 40 independent weight sets; the residual
    restarts from the same input every step; CUDA-graph replay."""
    import torch

    import bit_quantized_expert_gb300 as moe
    log(f"{wl.name}: generating {LAYERS} weight sets")
    layers = make_layers(wl, device, LAYERS)
    routers = []
    for l in range(LAYERS):
        r = synth.make_router(wl, seed=l)
        routers.append({k: torch.from_numpy(v.view(np.int16)).to(device) for k, v in r.items()})
    x0 = torch.randn((wl.T, wl.d), generator=torch.Generator(device=device).manual_seed(7), device=device)
    x = torch.empty_like(x0)
    h = torch.empty((wl.T, wl.d), dtype=torch.int16, device=device)
    lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device=device)
    y = torch.empty((wl.T, wl.d), dtype=torch.float32, device=device)
    dm = layers[0].dims(wl.T)
    ws = moe.alloc_workspace(dm, device)
    stream = torch.cuda.Stream(device=device)

    def step():
        x.copy_(x0)
        for l in range(LAYERS):
            moe.rmsnorm_router(dm, x, y if l > 0 else None, routers[l]["gamma"], routers[l]["w_router"], 1e-6,
                               h, lg, ws)
            layers[l].forward(h, lg, y, ws)

    with on_stream(stream):
        step()
    stream.synchronize()
    g = capture(step, stream)
    with on_stream(stream):
        g.replay()
    stream.synchronize()
    ms = timed_graph_steps(g, 1, g, steps, stream)
    log(f"{wl.name}: {ms / steps * 1e3:.1f} us per step")
    flags = moe.read_error_flags(ws)
    step_s = ms / 1e3 / steps
    # Every expert is touched at T = 2048.  Per layer: the layer's own algorithmic bytes (weights, its
    # input h, the logits, y) and the router weights.  The fp32 residual update and the writes of h and
    # the logits between layers are implementation overhead, not counted.
    per_layer = layer_bytes(wl, wl.T, wl.E) + wl.E * wl.d * 2
    flops = LAYERS * (layer_flops(wl, wl.T) + 2 * wl.T * wl.d * wl.E)
    out = {"workload": wl.name, "value": wl.T / step_s, "unit": "tokens/s (through 40 layers)",
           "ms_per_step": ms / steps, "steps": steps, "weight_sets": LAYERS, "flags": flags,
           "hbm": {"achieved": LAYERS * per_layer / step_s / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                   "frac": LAYERS * per_layer / step_s / 1e9 / pk["hbm_gbs"],
                   "algorithmic_bytes": LAYERS * per_layer},
           "tensor": {"achieved": flops / step_s / 1e12, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                      "frac": flops / step_s / 1e12 / pk["bf16_tflops"], "algorithmic_flops": flops},
           # per layer: rmsnorm, router GEMM and the eight kernels of a layer call; one residual copy
           "gpu_launches_per_step": LAYERS * 10}
    del layers, routers
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------------ CPU oracle

def attention_bytes(wl):
    """Algorithmic bytes of one decode-attention call: the keys and values of N positions for every
    key/value head (bf16), the bf16 query heads and the fp32 output."""
    return 2 * wl.Hkv * wl.N * wl.D * 2 + wl.Hq * wl.D * 2 + wl.Hq * wl.D * 4


def attention_bench(wl, steps, device, pk):
    """One step = one decode token through the model's ten full-attention layers at context N: each
    layer has its own bf16 key/value cache (10 x N x 1 KB in HBM, larger than L2, so no layer's
    cache is in L2 when it runs) and its own query; one library call per layer; CUDA-graph replay."""
    import torch

    import bit_quantized_expert_gb300 as moe
    log(f"{wl.name}: generating {wl.layers} caches")
    layers = [synth.torch_make_attention(wl.Hq, wl.Hkv, wl.D, wl.N, seed=l, device=device) for l in range(wl.layers)]
    gd = moe.gqa_dims(wl.Hq, wl.Hkv, wl.D, wl.N)
    ws = moe.alloc_gqa_workspace(gd, device)
    o = torch.empty((wl.layers, wl.Hq, wl.D), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device=device)

    def step():
        for l, c in enumerate(layers):
            moe.gqa_decode_attention(gd, c["q"], c["k"], c["v"], o[l], ws)

    with on_stream(stream):
        for _ in range(3):
            step()
    stream.synchronize()
    g = capture(step, stream)
    with on_stream(stream):
        for _ in range(3):
            g.replay()
    stream.synchronize()
    ms = timed_graph_steps(g, 1, g, steps, stream)
    # The same calls with a one-element torch kernel between them: it does not allow an early start,
    # so each call's copies begin only after the previous call has finished (no overlap across
    # calls); the separators' own time, measured alone, is subtracted.
    sep = torch.zeros(1, device=device)

    def step_sep():
        for l, c in enumerate(layers):
            sep.add_(1.0)
            moe.gqa_decode_attention(gd, c["q"], c["k"], c["v"], o[l], ws)

    def seps():
        for _ in range(wl.layers):
            sep.add_(1.0)

    with on_stream(stream):
        step_sep()
    stream.synchronize()
    g_sep, g_seps = capture(step_sep, stream), capture(seps, stream)
    with on_stream(stream):
        for _ in range(3):
            g_sep.replay()
            g_seps.replay()
    stream.synchronize()
    ms_sep = timed_graph_steps(g_sep, 1, g_sep, steps, stream)
    ms_seps = timed_graph_steps(g_seps, 1, g_seps, steps, stream)
    flags = moe.read_error_flags(ws)
    step_s = ms / 1e3 / steps
    call_s = step_s / wl.layers
    iso_s = (ms_sep - ms_seps) / 1e3 / steps / wl.layers
    nbytes = attention_bytes(wl)
    log(f"{wl.name}: {call_s * 1e6:.2f} us per layer call ({iso_s * 1e6:.2f} us without overlap across calls)")
    out = {"workload": wl.name, "ms_per_step": ms / steps, "us_per_layer_call": call_s * 1e6, "steps": steps,
           "layers": wl.layers, "flags": flags,
           "value": 1.0 / step_s, "unit": "decode tokens/s through the attention layers",
           "hbm": {"achieved": nbytes / call_s / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                   "frac": nbytes / call_s / 1e9 / pk["hbm_gbs"], "algorithmic_bytes_per_call": nbytes,
                   "note": "per call: attn_block_kernel + attn_merge_kernel; peak is the measured copy rate"},
           "us_per_layer_call_no_overlap": iso_s * 1e6,
           "hbm_frac_no_overlap": nbytes / iso_s / 1e9 / pk["hbm_gbs"],
           "gpu_launches_per_step": 2 * wl.layers}
    del layers
    torch.cuda.empty_cache()
    return out


# fp32 FMA peak for the scan's roofline: 152 SMs x 128 fp32 lanes x 2 flops per FMA x the maximum SM
# clock (MEASURED_PEAKS.json "sm_max_mhz", 2070 MHz on this pool): 80.5 TFLOP/s.
def fp32_peak_tflops(pk):
    return 152 * 128 * 2 * pk.get("sm_max_mhz", 2070.0) * 1e6 / 1e12


def scan_bytes(wl):
    """Algorithmic bytes of one scan call: the state in and out (fp32), q, k, v (bf16), g and beta
    (fp32) and o (fp32)."""
    return 2 * wl.H * wl.D * wl.D * 4 + wl.T * wl.H * (3 * wl.D * 2 + 2 * 4 + wl.D * 4)


def scan_flops(wl):
    """Two 128-term dots and one 128-wide update per state row, token and head: 6 flops per state
    element per token."""
    return 6 * wl.T * wl.H * wl.D * wl.D


def scan_bench(wl, steps, device, pk):
    """One step = wl.layers scan calls (each layer with its own state, updated in place, and its own
    inputs), replayed as a CUDA graph; L2 is flushed (a 256 MB write) before every timed step, outside
    the timed region, so each step starts with the states and inputs in HBM."""
    import torch

    import bit_quantized_expert_gb300 as moe
    layers = [synth.torch_make_scan(wl.T, wl.H, wl.D, seed=l, device=device, fresh=wl.fresh) for l in range(wl.layers)]
    gd = moe.gdn_dims(wl.T, wl.H, wl.D, wl.D)
    ws = moe.alloc_gdn_workspace(gd, device)
    o = torch.empty((wl.layers, wl.T, wl.H, wl.D), dtype=torch.float32, device=device)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device=device)

    # A decode step (several layers, one token each): each layer's state was last written by its own
    # scan of the previous step, so it may be read before the preceding launch ends.
    early = wl.layers > 1

    def step():
        for l, c in enumerate(layers):
            moe.gdn_scan(gd, c["q"], c["k"], c["v"], c["g"], c["beta"], c["S0"], c["S0"], o[l], ws, early_state=early)

    with on_stream(stream):
        for _ in range(3):
            step()
    stream.synchronize()
    gr = capture(step, stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with on_stream(stream):
        for _ in range(3):
            gr.replay()
        for e0, e1 in ev:
            flush.fill_(1.0)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
    stream.synchronize()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev)
    flags = moe.read_error_flags(ws)
    step_s = ms / 1e3 / steps
    call_s = step_s / wl.layers
    nbytes, flops = scan_bytes(wl), scan_flops(wl)
    peak_f = fp32_peak_tflops(pk)
    log(f"{wl.name}: {call_s * 1e6:.2f} us per layer call")
    out = {"workload": wl.name, "ms_per_step": ms / steps, "us_per_layer_call": call_s * 1e6, "steps": steps,
           "layers": wl.layers, "flags": flags, "value": wl.T / call_s, "unit": "tokens/s per layer",
           "hbm": {"achieved": nbytes / call_s / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                   "frac": nbytes / call_s / 1e9 / pk["hbm_gbs"], "algorithmic_bytes_per_call": nbytes},
           "alu": {"achieved": flops / call_s / 1e12, "peak": peak_f, "unit": "TFLOP/s",
                   "frac": flops / call_s / 1e12 / peak_f, "algorithmic_flops_per_call": flops,
                   "note": "fp32 peak derived from 152 SMs x 128 lanes x 2 x max SM clock"},
           "l2": "flushed before every timed step",
           "gpu_launches_per_step": wl.layers}
    del layers
    torch.cuda.empty_cache()
    return out


def oracle_rate(budget_s: float, max_tokens: int | None = None):
    """The float64 oracle on decode tokens of one layer (its cost does not depend on the weights)."""
    from oracle import moe_oracle as O
    wl = synth.DECODE
    host = synth.make_layer(wl, seed=0)
    inp = synth.make_inputs(wl, T=NI)
    O.moe_token(inp["x"][0], inp["logits"][0], host, wl.k)   # warm
    n, t0 = 0, time.perf_counter()
    while True:
        i = n % NI
        O.moe_token(inp["x"][i], inp["logits"][i], host, wl.k)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_tokens is not None and n >= max_tokens):
            break
    return n, el


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def config(world):
    return {"workload": synth.DECODE.name, "layers_per_step": LAYERS, "weight_sets": LAYERS,
            "global_batch": 1 * world, "seq_len": 1,
            "l2": "not flushed; inputs larger than L2 (40 weight sets, 18.2 GB, cycled per step)",
            "parallelism": f"replicas{world}" if world > 1 else "single GPU"}


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    budget = 60.0
    n, el = oracle_rate(budget, max_tokens=LAYERS * max(1, args.steps))
    steps = max(1, n // LAYERS)
    value = n / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / max(1, n) * LAYERS,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config(1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                             "sample": f"{n} decode layer-tokens (one layer's weights) in {el:.1f} s; "
                                       f"bounded to {budget:.0f} s"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(args):
    """Eager launches (no CUDA graph) of one workload over a few weight sets, for ncu: every kernel
    of the path shows up as its own launch.  Holds at most a few GB on the device."""
    import torch

    import bit_quantized_expert_gb300 as moe
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    moe.load_library()
    if args.profile == "attention":
        run_profile_attention(args)
        return
    if args.profile == "scan":
        run_profile_scan(args)
        return
    wl = {"decode": synth.DECODE, "prefill": synth.PREFILL, "skewed": synth.SKEWED, "stack": synth.STACK}[args.profile]
    n = args.profile_sets
    layers = make_layers(wl, device, n)
    T = wl.T
    ins = [synth.torch_make_inputs(wl, seed=1000 + l, device=device, T=(NI if T == 1 else T)) for l in range(n)]
    dm = layers[0].dims(T)
    ws = moe.alloc_workspace(dm, device)
    y = torch.empty((T, wl.d), dtype=torch.float32, device=device)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    total = args.warmup + args.steps
    for s in range(total):
        l = s % n
        if T == 1:
            i = s % NI
            layers[l].forward(ins[l]["x"][i:i + 1], ins[l]["logits"][i:i + 1], y, ws)
        else:
            layers[l].forward(ins[l]["x"], ins[l]["logits"], y, ws, operands=args.profile_operands)
    torch.cuda.synchronize()
    flags = moe.read_error_flags(ws)
    print(json.dumps({"profile": wl.name, "calls": total, "weight_sets": n, "flags": flags,
                      "wall_s": time.perf_counter() - t0}), flush=True)


def run_profile_attention(args):
    """Eager decode-attention calls at context 32768 over `profile_sets` (at least 6) distinct caches,
    192 MB or more in all (larger than L2)."""
    import torch

    import bit_quantized_expert_gb300 as moe
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    moe.load_library()
    wl = synth.GQA_32K
    n = max(6, args.profile_sets)
    layers = [synth.torch_make_attention(wl.Hq, wl.Hkv, wl.D, wl.N, seed=l, device=device) for l in range(n)]
    gd = moe.gqa_dims(wl.Hq, wl.Hkv, wl.D, wl.N)
    ws = moe.alloc_gqa_workspace(gd, device)
    o = torch.empty((wl.Hq, wl.D), dtype=torch.float32, device=device)
    torch.cuda.synchronize()
    total = args.warmup + args.steps
    for s in range(total):
        c = layers[s % n]
        moe.gqa_decode_attention(gd, c["q"], c["k"], c["v"], o, ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile": wl.name, "calls": total, "caches": n, "flags": moe.read_error_flags(ws)}), flush=True)


def run_profile_scan(args):
    """Eager scan calls over a 512-token prompt (16 heads), cycling `profile_sets` input sets."""
    import torch

    import bit_quantized_expert_gb300 as moe
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    moe.load_library()
    wl = synth.SCAN_512
    n = max(2, args.profile_sets)
    sets = [synth.torch_make_scan(wl.T, wl.H, wl.D, seed=l, device=device, fresh=wl.fresh) for l in range(n)]
    gd = moe.gdn_dims(wl.T, wl.H)
    ws = moe.alloc_gdn_workspace(gd, device)
    o = torch.empty((wl.T, wl.H, wl.D), dtype=torch.float32, device=device)
    torch.cuda.synchronize()
    total = args.warmup + args.steps
    for s in range(total):
        c = sets[s % n]
        moe.gdn_scan(gd, c["q"], c["k"], c["v"], c["g"], c["beta"], c["S0"], c["S0"], o, ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile": wl.name, "calls": total, "sets": n, "flags": moe.read_error_flags(ws)}), flush=True)


def main():
    args = parse()
    if args.profile is not None:
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import bit_quantized_expert_gb300 as moe
    moe.load_library()
    pk = peaks()

    res = decode_bench(args, world, rank, local, device, pk)
    extras, attn, scan = [], None, None
    if not args.no_extras and rank == 0:
        extras.append(prefill_bench(synth.PREFILL, 48, device, pk))
        extras.append(prefill_bench(synth.SKEWED, 24, device, pk))
        extras.append(prefill_bench(synth.PREFILL, 48, device, pk, operands="bf16"))
        extras.append(prefill_bench(synth.SKEWED, 24, device, pk, operands="bf16"))
        extras.append(stack_bench(synth.STACK, 5, device, pk))
        attn = [attention_bench(w, 20, device, pk) for w in (synth.GQA_32K, synth.GQA_64K, synth.GQA_128K)]
        scan = [scan_bench(w, 10, device, pk) for w in (synth.SCAN_DECODE, synth.SCAN_512, synth.SCAN_2048)]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, el = oracle_rate(20.0)
        cpu = {"value": n / el, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
               "sample": f"{n} decode layer-tokens through one layer in {el:.1f} s (float64 numpy oracle)"}
    if rank == 0:
        line = {"metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; random weights)",
                "config": config(world), "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"],
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"], "error_flags": res["flags"],
                "decode_hot_l2": res.get("hot_l2"), "decode_e2e_staged": res.get("e2e_staged"),
                "decode_small_T": res.get("small_T"), "decode_loads_only": res.get("loads_only"),
                "prefill": extras, "gqa_decode_attention": attn, "deltanet_scan": scan}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
