#!/usr/bin/env python3
"""Benchmark of the routed MoE FFN forward on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl strata|reference]

Workloads (synthetic, seeded; shapes of a Qwen3.6-35B-A3B MoE layer: H=2048,
256 experts, top-8, I = Is = 512, int4 weights with one fp16 scale per 32
inputs, bf16 activations):
  decode1   (default) T=1 decode through 10 distinct layers (seeds 0..9); one
            step = one token through each of the 10 layers, in order, as one
            CUDA graph; 16 token variants per layer rotate between steps, so
            the touched experts change and the 4.56 GB of weights defeat L2.
  decode16  the same with T=16 (8 requests x 2 MTP tokens, cosine-0.9 pairs)
            and a Zipf(1.1) router bias.
  stack     one token (--tokens 1 or 4) through a 40-layer residual MoE stack
            (one moe_stack_forward call, 18.2 GB resident) as one CUDA graph.
  prefill   T=2048 prompt tokens through one layer with Zipf-skewed routing
            (the tensor-core grouped GEMMs).

Printed: one JSON line (rank 0).  value = tokens per second through one MoE
layer (decode1/decode16: layer-tokens / s; stack: tokens / s through all 40
layers; prefill: prompt tokens / s).  The roofline object is for the
dominant kernel, timed alone with CUDA events on its own stream (HBM-bound
for the decode kernels, tensor-bound for the prefill GEMM); the default
decode1 line also carries a "prefill" block with the T=2048 layer and its
gate/up GEMM's tensor roofline.  cpu_baseline is the C oracle on the host.
--impl reference times that oracle itself on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import gen  # noqa: E402

METRIC = "MoE decode tok/s & expert-weight HBM GB/s vs ~8 TB/s; prefill tok/s, TC util"
EXPERT_BYTES = None          # filled per dims
NOMINAL_HBM_GBS = 8000.0


def expert_bytes(d) -> int:
    H, I = d.hidden, d.inter
    return 2 * I * H // 2 + 2 * I * (H // 32) * 2 + H * I // 2 + H * (I // 32) * 2


def shared_bytes(d) -> int:
    H, Is = d.hidden, d.shared_inter
    return 2 * Is * H // 2 + 2 * Is * (H // 32) * 2 + H * Is // 2 + H * (Is // 32) * 2


def router_bytes(d) -> int:
    return (d.n_experts + 1) * d.hidden * 2


def gu_bytes(d, I) -> int:
    return 2 * I * d.hidden // 2 + 2 * I * (d.hidden // 32) * 2


def dn_bytes(d, I) -> int:
    return d.hidden * I // 2 + d.hidden * (I // 32) * 2


# ------------------------------------------------------------- environment
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class Control:
    """Host-side control plane of the replicas: barrier and max over ranks
    (gloo; no data-path collective: every rank runs its own replica)."""

    def __init__(self, world):
        self.world = world
        self.pg = None
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.dist = dist

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, v: float) -> float:
        if self.world == 1:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            self.dist.destroy_process_group()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unparsed"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def kernel_traffic(kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            j = json.load(f)
    except (OSError, ValueError):
        return None
    ent = j.get(kernel)
    if not ent:
        return None
    src = os.path.join(ROOT, "quantized_moe_expert_fwd_gb300", "csrc", ent["source"])
    try:
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    return ent["bytes_per_launch"] if digest == ent["sha256"] else None


# --------------------------------------------------------------- oracle leg
def oracle_sample(dims, planes_list, xs, budget_s: float):
    """Layer-tokens per second of the C oracle on the host cores: whole
    layer-token forwards (one token through one layer) until budget_s has
    passed (at least one)."""
    import oracle
    oracle.build()
    n = 0
    t0 = time.perf_counter()
    while True:
        li = n % len(planes_list)
        oracle.moe_forward(dims, planes_list[li], xs[li])
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    return n / dt, n, dt


# ------------------------------------------------------------ GPU workloads
def build_decode(args, dev):
    import torch
    import quantized_moe_expert_fwd_gb300 as q
    cfg = gen.CONFIGS["decode1" if args.workload == "decode1" else "decode16"]
    dims = cfg.dims
    T = cfg.tokens
    nl = args.layers
    planes, layers = [], []
    for s in range(nl):
        p = gen.draw_layer(dims, s, bias=cfg.bias, alpha=cfg.alpha)
        layers.append(q.DeviceLayer(p, dev))
        planes.append(p)
    nvar = args.variants
    xs = [[None] * nl for _ in range(nvar)]
    xbufs = []
    for v in range(nvar):
        for li in range(nl):
            r = gen.draw_tokens(dims, T, 1000 * v + li, cfg.token_kind)
            rt = torch.from_numpy(r).to(dev)
            x = torch.empty((T, dims.hidden), dtype=torch.int16, device=dev)
            q.moe_rmsnorm(rt, x)
            xs[v][li] = x
    outs = [torch.empty((T, dims.hidden), dtype=torch.int16, device=dev) for _ in range(nl)]
    return dims, T, planes, layers, xs, outs, cfg


def _touched_per_layer(q, dims, layers, xs, outs, ws, stream, ids_buf, nl, v0=0):
    n_act = []
    for li in range(nl):
        q.moe_layer_forward(dims, layers[li], xs[v0][li], outs[li], ws, ids=ids_buf,
                            stream=stream)
        stream.synchronize()
        n_act.append(len(np.unique(ids_buf.cpu().numpy())))
    return n_act


def decode_stages(q, dims, layers, xs, outs, ws, stream, ids_buf, nl, T, dev):
    """The three decode kernels, each timed alone over the layers: one graph
    of reps x layers launches a stage, a workspace per layer so every call
    sees its own layer's plan.  {name: (us a launch, weight bytes)}."""
    import torch
    wss = [q.make_workspace(dims, T, dev) for _ in range(nl)]
    v0 = 0
    with torch.cuda.stream(stream):
        for li in range(nl):
            q.moe_decode_route(dims, layers[li], xs[v0][li], wss[li], stream=stream)
            q.moe_decode_gate_up(dims, layers[li], xs[v0][li], wss[li], stream=stream)
            q.moe_decode_down_combine(dims, layers[li], T, outs[li], wss[li], stream=stream)
        stream.synchronize()
        n_act = _touched_per_layer(q, dims, layers, xs, outs, ws, stream, ids_buf, nl)
        stages = {
            "k_route": (lambda li: q.moe_decode_route(dims, layers[li], xs[v0][li], wss[li],
                                                      stream=stream),
                        lambda li: router_bytes(dims) + gu_bytes(dims, dims.shared_inter)),
            "k_gate_up": (lambda li: q.moe_decode_gate_up(dims, layers[li], xs[v0][li], wss[li],
                                                          stream=stream),
                          lambda li: n_act[li] * gu_bytes(dims, dims.inter)),
            "k_down": (lambda li: q.moe_decode_down_combine(dims, layers[li], T, outs[li],
                                                            wss[li], stream=stream),
                       lambda li: n_act[li] * dn_bytes(dims, dims.inter)
                       + dn_bytes(dims, dims.shared_inter)),
        }
        # each stage captured as one graph of reps x 10 launches, so host-side
        # call overhead does not leak into the per-launch time
        per_stage = {}
        reps = 50
        for name, (fn, nbytes) in stages.items():
            for li in range(nl):
                fn(li)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for r in range(reps):
                    for li in range(nl):
                        fn(li)
            g.replay()
            stream.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(4):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (4 * reps * nl)
            per_stage[name] = (us, sum(nbytes(li) for li in range(nl)) / nl)
    return per_stage, {k: round(v[0], 3) for k, v in per_stage.items()}


def tc_layer_stages(q, dims, layers, xs, outs, ws, stream, ids_buf, nl, reps=5):
    """Per-kernel durations of the tcgen05 layer (moe_layer_profile, events
    between the launches), averaged over the layers and reps; the weight-
    streaming kernels carry their weight bytes.  {name: (us, bytes)}."""
    n_act = _touched_per_layer(q, dims, layers, xs, outs, ws, stream, ids_buf, nl)
    acc = {}
    for _ in range(reps):
        for li in range(nl):
            prof = q.moe_layer_profile(dims, layers[li], xs[0][li], outs[li], ws, stream=stream)
            for k, v in prof.items():
                acc[k] = acc.get(k, 0.0) + v / (reps * nl)
    mean_act = sum(n_act) / nl
    weight_bytes = {
        "router_gemm": router_bytes(dims),
        "gemm_gate_up": mean_act * gu_bytes(dims, dims.inter) + gu_bytes(dims, dims.shared_inter),
        "gemm_down": mean_act * dn_bytes(dims, dims.inter) + dn_bytes(dims, dims.shared_inter),
    }
    per_stage = {k: (acc[k], b) for k, b in weight_bytes.items() if k in acc}
    return per_stage, {k: round(v, 3) for k, v in acc.items()}


def run_strata(args, rank, world, local, ctl):
    import torch
    import quantized_moe_expert_fwd_gb300 as q
    q.build.build()
    q.load()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    dims, T, planes, layers, xs, outs, cfg = build_decode(args, dev)
    nl = len(layers)
    ws = q.make_workspace(dims, T, dev)
    stream = torch.cuda.Stream(dev)
    nvar = len(xs)

    def step_calls(v):
        for li in range(nl):
            q.moe_layer_forward(dims, layers[li], xs[v][li], outs[li], ws, stream=stream)

    with torch.cuda.stream(stream):
        for v in range(nvar):
            step_calls(v)
        stream.synchronize()
        if q.moe_get_device_status(ws, stream) != q.STRATA_OK:
            raise RuntimeError("device status after first pass")
        graphs = []
        for v in range(nvar):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step_calls(v)
            graphs.append(g)
        # clocks up and stable before the measured warm-up
        t_end = time.time() + (0.0 if args.profile else 0.5)
        i = 0
        while time.time() < t_end:
            graphs[i % nvar].replay()
            i += 1
            if i % 64 == 0:
                stream.synchronize()
        stream.synchronize()

        clocks = ClockSampler(local)
        clocks.start()
        for i in range(args.warmup):
            graphs[i % nvar].replay()
        stream.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ctl.barrier()
        torch.cuda.synchronize(dev)
        clocks.mark_start()
        ev0.record(stream)
        for i in range(args.steps):
            graphs[(i + args.warmup) % nvar].replay()
        ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize(dev)
        clocks.mark_end()
        ctl.barrier()
        clocks.stop()
        ms_total = ev0.elapsed_time(ev1)
    ms_total = ctl.max(ms_total)
    st = q.moe_get_device_status(ws, stream)
    if st != q.STRATA_OK:
        raise RuntimeError(f"device status {q.strata_status_str(st)}")

    ms_step = ms_total / args.steps
    layer_tokens = args.steps * nl * T * world
    value = layer_tokens / (ms_total / 1e3)

    if args.profile:
        return {"profile": True, "ms_per_step": ms_step, "value": value}, None

    # touched-expert bytes per layer-forward, from the routing of every variant
    touched = 0
    ids_buf = torch.empty((T, dims.top_k), dtype=torch.int32, device=dev)
    for v in range(nvar):
        for li in range(nl):
            q.moe_layer_forward(dims, layers[li], xs[v][li], outs[li], ws, ids=ids_buf,
                                stream=stream)
            stream.synchronize()
            touched += len(np.unique(ids_buf.cpu().numpy()))
    mean_touched = touched / (nvar * nl)
    layer_bytes = mean_touched * expert_bytes(dims) + shared_bytes(dims) + router_bytes(dims)
    gbs = layer_bytes * nl / (ms_step / 1e3) / 1e9

    tc_path = T > q.moe_layer_decode_max_tokens()
    if tc_path:
        per_stage, kernels_us = tc_layer_stages(q, dims, layers, xs, outs, ws, stream, ids_buf, nl)
    else:
        per_stage, kernels_us = decode_stages(q, dims, layers, xs, outs, ws, stream, ids_buf, nl,
                                              T, dev)
    dom = max(per_stage, key=lambda k: per_stage[k][0])
    dom_us, dom_bytes = per_stage[dom]
    hbm_peak, _, peak_src = measured_peaks()
    achieved = dom_bytes / (dom_us / 1e6) / 1e9
    launches_per_layer = (7 if T <= 32 else 9) if tc_path else 3

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        xh = [torch.empty((T, dims.hidden), dtype=torch.int16).pin_memory() for _ in range(nl)]
        oh = [torch.empty((T, dims.hidden), dtype=torch.int16).pin_memory() for _ in range(nl)]
        xd = [torch.empty((T, dims.hidden), dtype=torch.int16, device=dev) for _ in range(nl)]
        for li in range(nl):
            xh[li].copy_(xs[0][li].cpu())
        k_e2e = max(10, min(args.steps, 500))
        with torch.cuda.stream(stream):
            for it in range(3 + k_e2e):
                if it == 3:
                    stream.synchronize()
                    ctl.barrier()
                    t0 = time.perf_counter()
                for li in range(nl):
                    xd[li].copy_(xh[li], non_blocking=True)
                for li in range(nl):
                    q.moe_layer_forward(dims, layers[li], xd[li], outs[li], ws, stream=stream)
                for li in range(nl):
                    oh[li].copy_(outs[li], non_blocking=True)
                stream.synchronize()
            dt = time.perf_counter() - t0
        dt = ctl.max(dt)
        e2e = {"value": k_e2e * nl * T * world / dt, "unit": "tok/s",
               "h2d_bytes_per_step": nl * T * dims.hidden * 2,
               "d2h_bytes_per_step": nl * T * dims.hidden * 2}

    result = {
        "metric": METRIC,
        "value": value,
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded random int4 weights and activations of the real shapes)",
        "config": {
            "workload": cfg.description,
            "tokens_per_call": T,
            "layers_per_step": nl,
            "value_unit": "layer-tokens per second (one token through one MoE layer)",
            "l2": f"inputs larger than L2: {nl} layers x 455.8 MB resident, "
                  f"{len(xs)} token variants per layer rotating between steps",
            "arithmetic": "int4 weights x bf16 activations, fp32 accumulate",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "expert_weight_gbs": gbs,
        "expert_weight_frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
        "touched_experts_per_layer": mean_touched,
        "roofline": {
            "kernel": dom,
            "bound": "hbm",
            "achieved": achieved,
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": achieved / hbm_peak,
            "peak_source": f"{peak_src} (burst copy, kernel timed alone)",
            "traffic": kernel_traffic(dom),
            "us_per_launch": dom_us,
            "algorithmic_bytes_per_launch": dom_bytes,
            "stages_us": {k: round(v[0], 3) for k, v in per_stage.items()},
        },
        "kernels": ("tcgen05 grouped GEMMs (T above the whole-layer decode switch)"
                    if tc_path else "decode kernels"),
        "kernels_us": kernels_us,
        "clocks": clocks.summary(),
        "e2e": e2e,
        "gpu_launches": args.steps * nl * launches_per_layer,
    }
    return result, (dims, planes, xs, nl)


def prefill_flops(d, T):
    H, E, K, I, Is = d.hidden, d.n_experts, d.top_k, d.inter, d.shared_inter
    routed = 2.0 * T * K * (2 * I * H + H * I)
    shared = 2.0 * T * (2 * Is * H + H * Is)
    router = 2.0 * T * (E + 1) * H
    return routed + shared + router, 2.0 * (T * K * 2 * I * H + T * 2 * Is * H)


def run_prefill(dev, reps=20, warmup=3):
    """Prefill T=2048 through one Zipf-routed layer: time per layer (CUDA
    graph), tokens/s, tensor-core FLOP rate, and the per-kernel split."""
    import torch
    import quantized_moe_expert_fwd_gb300 as q
    cfg = gen.CONFIGS["prefill"]
    dims, T = cfg.dims, cfg.tokens
    planes = gen.draw_layer(dims, 0, bias=cfg.bias, alpha=cfg.alpha)
    dl = q.DeviceLayer(planes, dev)
    r = torch.from_numpy(gen.draw_tokens(dims, T, 0, cfg.token_kind)).to(dev)
    x = torch.empty((T, dims.hidden), dtype=torch.int16, device=dev)
    q.moe_rmsnorm(r, x)
    out = torch.empty((T, dims.hidden), dtype=torch.int16, device=dev)
    ws = q.make_workspace(dims, T, dev)
    st = torch.cuda.Stream(dev)
    with torch.cuda.stream(st):
        q.moe_layer_forward(dims, dl, x, out, ws, stream=st)
        st.synchronize()
        if q.moe_get_device_status(ws, st) != q.STRATA_OK:
            raise RuntimeError("prefill: device status")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            q.moe_layer_forward(dims, dl, x, out, ws, stream=st)
        for _ in range(warmup):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            g.replay()
        e1.record(st)
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        prof = None
        for _ in range(3):
            prof = q.moe_layer_profile(dims, dl, x, out, ws, stream=st)
    total, gu_flops = prefill_flops(dims, T)
    _, bf16_peak, src = measured_peaks()
    gu_us = prof["gemm_gate_up"]
    return {
        "workload": cfg.description,
        "tokens": T,
        "us_per_layer": us,
        "tok_per_s": T / (us / 1e6),
        "tflops": total / (us / 1e6) / 1e12,
        "tc_frac_of_peak": total / (us / 1e6) / 1e12 / bf16_peak,
        "peak_tflops": bf16_peak,
        "peak_source": src,
        "kernels_us": {k: round(v, 2) for k, v in prof.items()},
        "gate_up_gemm": {"us": gu_us, "tflops": gu_flops / (gu_us / 1e6) / 1e12,
                         "frac": gu_flops / (gu_us / 1e6) / 1e12 / bf16_peak},
        "launches_per_layer": len(prof),
    }


def run_prefill_line(args, rank, world, local, ctl):
    """The prefill workload as the primary line: value = prompt tokens/s
    through one MoE layer at T=2048."""
    import torch
    import quantized_moe_expert_fwd_gb300 as q
    q.build.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if args.profile:
        # lean run for ncu: plain calls, no graphs, no oracle
        cfg = gen.CONFIGS["prefill"]
        dims, T = cfg.dims, cfg.tokens
        dl = q.DeviceLayer(gen.draw_layer(dims, 0, bias=cfg.bias, alpha=cfg.alpha), dev)
        r = torch.from_numpy(gen.draw_tokens(dims, T, 0, cfg.token_kind)).to(dev)
        x = torch.empty((T, dims.hidden), dtype=torch.int16, device=dev)
        q.moe_rmsnorm(r, x)
        out = torch.empty((T, dims.hidden), dtype=torch.int16, device=dev)
        ws = q.make_workspace(dims, T, dev)
        for _ in range(args.warmup + args.steps):
            q.moe_layer_forward(dims, dl, x, out, ws)
        torch.cuda.synchronize()
        return {"profile": True, "status": q.moe_get_device_status(ws)}
    clocks = ClockSampler(local)
    clocks.start()
    pf = run_prefill(dev, reps=args.steps, warmup=args.warmup)
    clocks.stop()
    us = ctl.max(pf["us_per_layer"])
    total, _ = prefill_flops(gen.CONFIGS["prefill"].dims, pf["tokens"])
    hbm, peak, src = measured_peaks()
    line = {
        "metric": METRIC,
        "value": pf["tokens"] * world / (us / 1e6),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": us / 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded random int4 weights and activations of the real shapes)",
        "config": {"workload": pf["workload"], "tokens_per_call": pf["tokens"],
                   "value_unit": "prompt tokens per second through one MoE layer",
                   "l2": "inputs larger than L2: 455.8 MB of weights read per step",
                   "arithmetic": "int4 weights dequantised to fp16 x fp16 activations on "
                                 "tcgen05, fp32 accumulate"},
        "roofline": {"kernel": "k_pf_gemm_sab<gate/up>", "bound": "tensor",
                     "achieved": pf["gate_up_gemm"]["tflops"], "peak": peak,
                     "unit": "TFLOP/s", "frac": pf["gate_up_gemm"]["frac"],
                     "peak_source": f"{src} bf16 (fp16 runs at the same rate), burst",
                     "traffic": kernel_traffic("k_pf_gemm_gate_up"),
                     "us_per_launch": pf["gate_up_gemm"]["us"]},
        "tc_frac_whole_layer": pf["tc_frac_of_peak"],
        "kernels_us": pf["kernels_us"],
        "clocks": clocks.summary(),
        "gpu_launches": args.steps * pf["launches_per_layer"],
        "cpu_baseline": None,
        "e2e": None,
    }
    return line


def run_stack_line(args, rank, world, local, ctl):
    """One decode step of T tokens through the 40-layer residual MoE stack
    (moe_block_forward x 40 in one CUDA graph): value = tokens/s through the
    whole stack."""
    import torch
    import quantized_moe_expert_fwd_gb300 as q
    q.build.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    cfg = gen.CONFIGS["stack"]
    dims, T = cfg.dims, args.tokens
    layers = []
    for s in cfg.seeds:
        layers.append(q.DeviceLayer(gen.draw_layer(dims, s), dev))
    nvar = args.variants
    r0s = [torch.from_numpy(gen.draw_tokens(dims, T, 5000 + v, "resid")).to(dev)
           for v in range(nvar)]
    resid = torch.empty((T, dims.hidden), dtype=torch.float32, device=dev)
    ws = q.make_workspace(dims, T, dev)
    st = torch.cuda.Stream(dev)
    ids = torch.empty((T, dims.top_k), dtype=torch.int32, device=dev)

    def step(v):
        resid.copy_(r0s[v])
        q.moe_stack_forward(dims, layers, resid, ws, stream=st)

    with torch.cuda.stream(st):
        step(0)
        st.synchronize()
        if q.moe_get_device_status(ws, st) != q.STRATA_OK:
            raise RuntimeError("stack: device status")
        graphs = []
        for v in range(nvar):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                step(v)
            graphs.append(g)
        for i in range(max(args.warmup, 3)):
            graphs[i % nvar].replay()
        st.synchronize()
        clocks = ClockSampler(local)
        clocks.start()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        ctl.barrier()
        torch.cuda.synchronize(dev)
        e0.record(st)
        for i in range(args.steps):
            graphs[i % nvar].replay()
        e1.record(st)
        e1.synchronize()
        ctl.barrier()
        clocks.stop()
        ms = ctl.max(e0.elapsed_time(e1)) / args.steps
        # touched experts per layer (routing of variant 0 through the stack)
        resid.copy_(r0s[0])
        touched = 0
        xo = torch.empty((T, dims.hidden), dtype=torch.int16, device=dev)
        for dl in layers:
            q.moe_block_forward(dims, dl, resid, ws, x_out=xo, stream=st)
            q.moe_route(dims, dl, xo, ids, torch.empty((T, dims.top_k), device=dev),
                        torch.empty((T,), device=dev), ws, stream=st)
            st.synchronize()
            touched += len(np.unique(ids.cpu().numpy()))
    nl = len(layers)
    step_bytes = touched * expert_bytes(dims) + nl * (shared_bytes(dims) + router_bytes(dims))
    gbs = step_bytes / (ms / 1e3) / 1e9
    hbm, _, src = measured_peaks()
    # per step: the residual reset (a copy kernel) and each layer's kernels
    # (rmsnorm + 3 decode kernels, or rmsnorm + 7 / 9 tcgen05-path kernels)
    launches = 1 + nl * (4 if T <= q.moe_layer_decode_max_tokens() else (8 if T <= 32 else 10))
    return {
        "metric": METRIC,
        "value": T * world / (ms / 1e3),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded random int4 weights and activations of the real shapes)",
        "config": {"workload": f"{cfg.description}; T={T}", "tokens_per_call": T,
                   "layers_per_step": nl,
                   "value_unit": "tokens per second through the whole 40-layer stack",
                   "l2": "inputs larger than L2: 18.2 GB of weights resident, "
                         f"{nvar} token variants rotating"},
        "expert_weight_gbs": gbs,
        "expert_weight_frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
        "hbm_frac_of_measured": gbs / hbm,
        "us_per_layer": ms * 1e3 / nl,
        "clocks": clocks.summary(),
        "gpu_launches": args.steps * launches,
        "cpu_baseline": None,
        "e2e": None,
    }


def cpu_baseline_block(dims, planes, xs_dev, nl, budget):
    import torch
    xs = [xs_dev[0][li].cpu().numpy().view(np.uint16) for li in range(nl)]
    v, n, dt = oracle_sample(dims, planes, xs, budget)
    return {"value": v, "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} layer-token forwards (T=1, layers cycling over seeds 0..9) "
                      f"in {dt:.1f} s, OpenMP over experts"}


def run_reference(args, rank, world):
    """The CPU oracle, as it stands, on the host cores: each step one
    layer-token forward of the same workload."""
    import oracle
    oracle.build()
    cfg = gen.CONFIGS["decode1" if args.workload == "decode1" else "decode16"]
    dims = cfg.dims
    nl = 10
    planes = [gen.draw_layer(dims, s, bias=cfg.bias, alpha=cfg.alpha) for s in range(nl)]
    xs = [oracle.rmsnorm(gen.draw_tokens(dims, cfg.tokens, li, cfg.token_kind))
          for li in range(nl)]
    # size the steps so the whole run stays within a few minutes
    t0 = time.perf_counter()
    oracle.moe_forward(dims, planes[0], xs[0])
    t_step = time.perf_counter() - t0
    budget = 150.0
    k = args.steps
    if (args.steps + args.warmup) * t_step > budget:
        k = max(3, int(budget / t_step) - args.warmup)
    for i in range(args.warmup):
        oracle.moe_forward(dims, planes[i % nl], xs[i % nl])
    t0 = time.perf_counter()
    for i in range(k):
        oracle.moe_forward(dims, planes[i % nl], xs[i % nl])
    dt = time.perf_counter() - t0
    value = k * cfg.tokens / dt
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tok/s",
        "n_gpus": world,
        "steps": k,
        "steps_requested": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt / k * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded random int4 weights and activations of the real shapes)",
        "config": {"workload": cfg.description, "tokens_per_call": cfg.tokens,
                   "value_unit": "layer-tokens per second (one token through one MoE layer)"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{k} layer-token forwards of the C oracle (fp32, "
                                   f"OpenMP over experts) in {dt:.1f} s"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["strata", "reference"], default="strata")
    ap.add_argument("--workload", choices=["decode1", "decode16", "prefill", "stack"],
                    default="decode1")
    ap.add_argument("--tokens", type=int, default=1, help="stack workload: tokens per step")
    ap.add_argument("--variants", type=int, default=16)
    ap.add_argument("--layers", type=int, default=10)
    ap.add_argument("--profile", action="store_true",
                    help="lean run for ncu: no clock warm loop, stage timing, e2e or oracle")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="leave out the prefill (T=2048) block of the line")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    ctl = Control(world)
    if args.workload == "stack":
        try:
            line = run_stack_line(args, rank, world, local, ctl)
            if rank == 0:
                print(json.dumps(line), flush=True)
        finally:
            ctl.close()
        return
    if args.workload == "prefill":
        try:
            print_line = run_prefill_line(args, rank, world, local, ctl)
            if rank == 0 and print_line is not None:
                print(json.dumps(print_line), flush=True)
        finally:
            ctl.close()
        return
    try:
        result, extra = run_strata(args, rank, world, local, ctl)
        if extra is None:
            if rank == 0:
                print(json.dumps(result), flush=True)
            return
        dims, planes, xs, nl = extra
        if rank == 0 and world == 1 and not args.no_prefill:
            # the prefill configuration beside the decode line: T=2048 through
            # one layer, tensor-core rate of the gate/up GEMM
            import torch
            pf = run_prefill(torch.device(f"cuda:{local}"), reps=20, warmup=3)
            result["prefill"] = {
                "workload": pf["workload"], "tokens": pf["tokens"],
                "tok_per_s": pf["tok_per_s"], "us_per_layer": pf["us_per_layer"],
                "roofline": {"kernel": "k_pf_gemm_sab<gate/up>", "bound": "tensor",
                             "achieved": pf["gate_up_gemm"]["tflops"],
                             "peak": pf["peak_tflops"], "unit": "TFLOP/s",
                             "frac": pf["gate_up_gemm"]["frac"],
                             "peak_source": pf["peak_source"],
                             "traffic": kernel_traffic("k_pf_gemm_gate_up"),
                             "us_per_launch": pf["gate_up_gemm"]["us"]},
                "tc_frac_whole_layer": pf["tc_frac_of_peak"],
                "kernels_us": pf["kernels_us"],
            }
        if rank == 0:
            if world == 1 and args.cpu_budget > 0:
                result["cpu_baseline"] = cpu_baseline_block(dims, planes, xs, nl,
                                                            args.cpu_budget)
            else:
                result["cpu_baseline"] = None
            print(json.dumps(result), flush=True)
    finally:
        ctl.close()


if __name__ == "__main__":
    main()
