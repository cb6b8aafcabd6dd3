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
  stack     T tokens (--tokens 1 or 4) through a 40-layer residual MoE stack
            (one moe_stack_forward call, 18.2 GB resident) as one CUDA graph,
            16 residual variants rotating.
  prefill   T=2048 prompt tokens through one layer with Zipf-skewed routing
            (the tensor-core grouped GEMMs).

Printed: one JSON line (rank 0).  value = tokens per second through one MoE
layer (decode1/decode16: layer-tokens / s; stack: tokens / s through all 40
layers; prefill: prompt tokens / s).  The default decode1 line also carries
"decode16", "stack_t1", "stack_t4" and "prefill" blocks, each with its own
roofline: HBM-bound for the decode kernels (the persistent decode kernel is
the whole layer; on the tensor-core path, the gate/up GEMM that streams the
weights), tensor-bound for the prefill GEMM.  Clocks are sampled with NVML
(read-only queries) during every timed region.  cpu_baseline is the C oracle
on the host cores, one thread and all of them.  --impl reference times that
oracle itself on the same workload, token seeds and metric.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import platform
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import gen  # noqa: E402

METRIC = "MoE decode tok/s & expert-weight HBM GB/s vs ~8 TB/s; prefill tok/s, TC util"
NOMINAL_HBM_GBS = 8000.0
N_LAYERS = 10            # distinct layers of the decode workloads
N_STACK = 40


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


def token_seed(variant: int, layer: int) -> int:
    """Seed of the tokens of one (variant, layer) of the decode workloads."""
    return 1000 * variant + layer


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
    """SM clock and clock-event (throttle) reasons of one GPU, sampled every
    20 ms by a thread through NVML's read-only queries, kept for the marked
    (timed) windows."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        self.dev = torch_device
        self.samples = []          # (time, sm MHz, reasons bits)
        self.windows = []
        self.max_mhz = None
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._h = None

    def _open(self):
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        bus = None
        try:
            import torch
            p = torch.cuda.get_device_properties(self.dev)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except (AttributeError, RuntimeError):
            bus = None
        ok = bus is not None and nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(),
                                                                      ctypes.byref(h)) == 0
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(self.dev.index or 0, ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._nvml, self._h = nv, h

    def _run(self):
        nv, h = self._nvml, self._h
        mhz = ctypes.c_uint()
        bits = ctypes.c_ulonglong()
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and \
                    fn(h, ctypes.byref(bits)) == 0:
                self.samples.append((time.time(), float(mhz.value), int(bits.value)))
            self._stop.wait(0.02)

    def start(self):
        try:
            self._open()
        except OSError as e:
            self.error = str(e)
            return self
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        return self

    def mark(self):
        """Context manager around a timed region."""
        sampler = self

        class _Win:
            def __enter__(self):
                self.t0 = time.time()
                return self

            def __exit__(self, *exc):
                sampler.windows.append((self.t0, time.time()))
                return False
        return _Win()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)
            self._thread = None
            try:
                self._nvml.nvmlShutdown()
            except OSError:
                pass

    def summary(self):
        if self.error is not None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"],
                    "samples": 0, "source": self.error}
        inside = [s for s in self.samples
                  if any(t0 <= s[0] <= t1 for t0, t1 in self.windows)] or self.samples
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"],
                    "samples": 0, "source": "nvml"}
        reasons = set()
        for _, _, bits in inside:
            for b, name in self.REASONS.items():
                if bits & b:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(inside),
                "source": "nvml, 20 ms, timed regions only"}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return (float(j["hbm_gbs"]), float(j["bf16_tflops"]),
                float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured")
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


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


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            txt = f.read()
    except OSError:
        return platform.machine()
    for line in txt.splitlines():
        if line.startswith("model name"):
            return line.split(":", 1)[1].strip()
    parts = {}
    for line in txt.splitlines():
        if ":" in line:
            k, v = (x.strip() for x in line.split(":", 1))
            parts.setdefault(k, v)
    return (f"{platform.machine()} (CPU implementer {parts.get('CPU implementer', '?')}, "
            f"part {parts.get('CPU part', '?')})")


# -------------------------------------------------------------- GPU set-up
def draw_layers(dims, seeds):
    """gen.draw_layer over the seeds, in order, drawn on a few threads at a
    time (numpy's generators release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    seeds = list(seeds)
    nt = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(nt) as ex:
        for i in range(0, len(seeds), nt):
            yield from ex.map(lambda s: gen.draw_layer(dims, s), seeds[i:i + nt])


class Resident:
    """The workloads' layers resident on the GPU (seeds 0..n-1, drawn once),
    and the host planes of the first N_LAYERS for the CPU oracle."""

    def __init__(self, dev, n):
        import quantized_moe_expert_fwd_gb300 as q
        self.dev = dev
        self.dims = gen.QWEN
        self.layers = []
        self.planes = []
        for p in draw_layers(self.dims, range(n)):
            self.layers.append(q.DeviceLayer(p, dev))
            if len(self.planes) < N_LAYERS:
                self.planes.append(p)

    def biased(self, n, alpha):
        return [dl.with_bias(gen.zipf_bias(self.dims.n_experts, alpha, s), self.dev)
                for s, dl in enumerate(self.layers[:n])]


def replay_timed(graphs, steps, warmup, stream, ctl, clocks):
    """Replays graphs[i % len] for warmup then `steps` timed steps (barrier +
    synchronize on both sides, CUDA events on `stream`); ms a step, max over
    ranks."""
    import torch
    for i in range(max(warmup, 3)):
        graphs[i % len(graphs)].replay()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    ctl.barrier()
    torch.cuda.synchronize()
    with clocks.mark():
        e0.record(stream)
        for i in range(steps):
            graphs[(i + warmup) % len(graphs)].replay()
        e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
    ctl.barrier()
    return ctl.max(e0.elapsed_time(e1)) / steps


def launches_per_layer(q, dims, T):
    path = q.moe_layer_path(dims, T)
    if path == q.PATH_PERSISTENT:
        return 1
    if path == q.PATH_DECODE:
        return 3
    return 7 if T <= 32 else 9


def decode_block(q, res, T, kind, bias_alpha, args, ctl, clocks, stream, want_e2e=False):
    """A decode workload: T tokens through each of args.layers layers a step,
    16 token variants rotating.  Returns the block's dict."""
    import torch
    dev, dims = res.dev, res.dims
    nl = args.layers
    layers = res.layers[:nl] if bias_alpha is None else res.biased(nl, bias_alpha)
    nvar = args.variants
    xs = [[None] * nl for _ in range(nvar)]
    for v in range(nvar):
        for li in range(nl):
            r = torch.from_numpy(gen.draw_tokens(dims, T, token_seed(v, li), kind)).to(dev)
            x = torch.empty((T, dims.hidden), dtype=torch.int16, device=dev)
            q.moe_rmsnorm(r, x, stream=stream)
            xs[v][li] = x
    outs = [torch.empty((T, dims.hidden), dtype=torch.int16, device=dev) for _ in range(nl)]
    ws = q.make_workspace(dims, T, dev)

    def step(v):
        for li in range(nl):
            q.moe_layer_forward(dims, layers[li], xs[v][li], outs[li], ws, stream=stream)

    with torch.cuda.stream(stream):
        for v in range(nvar):
            step(v)
        stream.synchronize()
        if q.moe_get_device_status(ws, stream) != q.STRATA_OK:
            raise RuntimeError(f"decode T={T}: device status after the first pass")
        graphs = []
        for v in range(nvar):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(v)
            graphs.append(g)
        # clocks up before the measured warm-up
        t_end = time.time() + 0.5
        i = 0
        while time.time() < t_end:
            graphs[i % nvar].replay()
            i += 1
            if i % 64 == 0:
                stream.synchronize()
        stream.synchronize()
        ms_step = replay_timed(graphs, args.steps, args.warmup, stream, ctl, clocks)
        if q.moe_get_device_status(ws, stream) != q.STRATA_OK:
            raise RuntimeError(f"decode T={T}: device status after the timed steps")
        # touched experts per layer-forward, over every (variant, layer)
        ids = torch.empty((T, dims.top_k), dtype=torch.int32, device=dev)
        touched = []
        for v in range(nvar):
            for li in range(nl):
                q.moe_layer_forward(dims, layers[li], xs[v][li], outs[li], ws, ids=ids,
                                    stream=stream)
                stream.synchronize()
                touched.append(len(np.unique(ids.cpu().numpy())))
        mean_touched = float(np.mean(touched))
        layer_bytes = mean_touched * expert_bytes(dims) + shared_bytes(dims) + router_bytes(dims)
        layer_us = ms_step * 1e3 / nl
        hbm, _, _, src = measured_peaks()
        path = q.moe_layer_path(dims, T)
        if path == q.PATH_PERSISTENT:
            # one kernel is the whole layer: its bytes are the layer's
            roof = {"kernel": "k_persist (the whole layer, one launch)", "bound": "hbm",
                    "achieved": layer_bytes / (layer_us / 1e6) / 1e9, "peak": hbm,
                    "unit": "GB/s", "traffic": kernel_traffic("k_persist@decode_T1"),
                    "us_per_launch": layer_us, "algorithmic_bytes_per_launch": layer_bytes,
                    "peak_source": f"{src} HBM copy bandwidth (burst)",
                    "timing": "CUDA events over the timed graph replays, per layer"}
        else:
            # the kernels one at a time (events between launches), variants
            # and layers rotating; the gate/up GEMM streams the routed and
            # shared gate/up weights
            acc, n = {}, 0
            for v in range(nvar):
                for li in range(nl):
                    prof = q.moe_layer_profile(dims, layers[li], xs[v][li], outs[li], ws,
                                               stream=stream)
                    for k, u in prof.items():
                        acc[k] = acc.get(k, 0.0) + u
                    n += 1
            kus = {k: round(u / n, 3) for k, u in acc.items()}
            gu_us = kus["gemm_gate_up"]
            gbytes = mean_touched * gu_bytes(dims, dims.inter) + gu_bytes(dims, dims.shared_inter)
            roof = {"kernel": "k_pf_gemm_sab<gate/up>", "bound": "hbm",
                    "achieved": gbytes / (gu_us / 1e6) / 1e9, "peak": hbm, "unit": "GB/s",
                    "traffic": kernel_traffic("k_pf_gemm_sab<1>@decode_T16"),
                    "us_per_launch": gu_us,
                    "algorithmic_bytes_per_launch": gbytes,
                    "peak_source": f"{src} HBM copy bandwidth (burst)",
                    "timing": "moe_layer_profile: events between the kernels, "
                              f"{n} layer calls rotating", "kernels_us": kus}
        roof["frac"] = roof["achieved"] / roof["peak"]
        block = {"tokens": T, "value": nl * T / (ms_step / 1e3), "unit": "layer-tok/s",
                 "ms_per_step": ms_step, "us_per_layer": layer_us,
                 "touched_experts_per_layer": mean_touched,
                 "expert_weight_gbs": layer_bytes / (layer_us / 1e6) / 1e9,
                 "path": {1: "persistent", 2: "decode kernels", 3: "tcgen05"}.get(path, "?"),
                 "roofline": roof, "gpu_launches_per_step": nl * launches_per_layer(q, dims, T)}
        block["expert_weight_frac_of_8tbs"] = block["expert_weight_gbs"] / NOMINAL_HBM_GBS
        if want_e2e:
            # end to end through the public call with host buffers: every step
            # copies its tokens in from pinned memory and its outputs back
            xh = [[xs[v][li].cpu().pin_memory() for li in range(nl)] for v in range(nvar)]
            oh = [torch.empty((T, dims.hidden), dtype=torch.int16).pin_memory() for _ in range(nl)]
            xd = [torch.empty((T, dims.hidden), dtype=torch.int16, device=dev) for _ in range(nl)]
            k_e2e = max(10, min(args.steps, 500))
            for it in range(3 + k_e2e):
                if it == 3:
                    stream.synchronize()
                    ctl.barrier()
                    t0 = time.perf_counter()
                v = it % nvar
                for li in range(nl):
                    xd[li].copy_(xh[v][li], non_blocking=True)
                for li in range(nl):
                    q.moe_layer_forward(dims, layers[li], xd[li], outs[li], ws, stream=stream)
                for li in range(nl):
                    oh[li].copy_(outs[li], non_blocking=True)
                stream.synchronize()
            dt = ctl.max(time.perf_counter() - t0)
            block["e2e"] = {"value": k_e2e * nl * T * ctl.world / dt, "unit": "tok/s",
                            "h2d_bytes_per_step": nl * T * dims.hidden * 2,
                            "d2h_bytes_per_step": nl * T * dims.hidden * 2}
        block["_xs"] = xs
    return block


def stack_block(q, res, T, args, ctl, clocks, stream, steps=None):
    """T tokens through the 40-layer residual stack, one moe_stack_forward a
    step, 16 residual variants rotating."""
    import torch
    dev, dims = res.dev, res.dims
    layers = res.layers[:N_STACK]
    nvar = args.variants
    r0s = [torch.from_numpy(gen.draw_tokens(dims, T, 5000 + v, "resid")).to(dev)
           for v in range(nvar)]
    resid = torch.empty((T, dims.hidden), dtype=torch.float32, device=dev)
    ws = q.make_workspace(dims, T, dev)

    def step(v):
        resid.copy_(r0s[v])
        q.moe_stack_forward(dims, layers, resid, ws, stream=stream)

    with torch.cuda.stream(stream):
        step(0)
        stream.synchronize()
        if q.moe_get_device_status(ws, stream) != q.STRATA_OK:
            raise RuntimeError(f"stack T={T}: device status")
        graphs = []
        for v in range(nvar):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(v)
            graphs.append(g)
        if steps is None:
            steps = max(20, min(args.steps // 10, 300))
        ms = replay_timed(graphs, steps, args.warmup, stream, ctl, clocks)
        if q.moe_get_device_status(ws, stream) != q.STRATA_OK:
            raise RuntimeError(f"stack T={T}: device status after the timed steps")
        # touched experts of every layer, for variant 0
        resid.copy_(r0s[0])
        touched = 0
        ids = torch.empty((T, dims.top_k), dtype=torch.int32, device=dev)
        xo = torch.empty((T, dims.hidden), dtype=torch.int16, device=dev)
        for dl in layers:
            q.moe_block_forward(dims, dl, resid, ws, x_out=xo, stream=stream)
            q.moe_route(dims, dl, xo, ids, torch.empty((T, dims.top_k), device=dev),
                        torch.empty((T,), device=dev), ws, stream=stream)
            stream.synchronize()
            touched += len(np.unique(ids.cpu().numpy()))
    nl = len(layers)
    step_bytes = touched * expert_bytes(dims) + nl * (shared_bytes(dims) + router_bytes(dims))
    hbm, _, _, src = measured_peaks()
    path = q.moe_layer_path(dims, T)
    if path == q.PATH_PERSISTENT:
        per_layer = kernel_traffic("k_persist@decode_T1")
        roof = {"kernel": f"k_persist (the {nl}-layer stack, one launch)", "bound": "hbm",
                "achieved": step_bytes / (ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                "traffic": None if per_layer is None else per_layer * nl,
                "traffic_note": "the one-layer T=1 capture's DRAM bytes x layers (a T=1 layer "
                                "touches 8 experts whatever the token)" if T == 1 else None,
                "us_per_launch": ms * 1e3, "algorithmic_bytes_per_launch": step_bytes,
                "peak_source": f"{src} HBM copy bandwidth (burst)"}
        launches = 1            # the kernel (the residual reset is a torch copy)
    else:
        roof = {"kernel": f"all kernels of the {nl} layers (step)", "bound": "hbm",
                "achieved": step_bytes / (ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                "traffic": None, "us_per_launch": ms * 1e3,
                "algorithmic_bytes_per_launch": step_bytes,
                "peak_source": f"{src} HBM copy bandwidth (burst)"}
        launches = nl * (1 + launches_per_layer(q, dims, T))
    roof["frac"] = roof["achieved"] / roof["peak"]
    return {"tokens": T, "value": T * ctl.world / (ms / 1e3), "unit": "tok/s",
            "ms_per_step": ms, "steps": steps, "us_per_layer": ms * 1e3 / nl,
            "touched_experts_per_step": touched,
            "expert_weight_gbs": step_bytes / (ms / 1e3) / 1e9,
            "path": {1: "persistent", 2: "decode kernels", 3: "tcgen05"}.get(path, "?"),
            "roofline": roof, "gpu_launches_per_step": launches}


def prefill_flops(d, T):
    H, E, K, I, Is = d.hidden, d.n_experts, d.top_k, d.inter, d.shared_inter
    routed = 2.0 * T * K * (2 * I * H + H * I)
    shared = 2.0 * T * (2 * Is * H + H * Is)
    router = 2.0 * T * (E + 1) * H
    return routed + shared + router, 2.0 * (T * K * 2 * I * H + T * 2 * Is * H)


def prefill_block(q, res, args, ctl, clocks, stream, reps=20):
    """T=2048 through one Zipf-routed layer: time per layer (CUDA graph),
    tokens/s, the gate/up GEMM's tensor rate, and the per-kernel split."""
    import torch
    cfg = gen.CONFIGS["prefill"]
    dims, T = cfg.dims, cfg.tokens
    dl = res.layers[0].with_bias(gen.zipf_bias(dims.n_experts, cfg.alpha, 0), res.dev)
    r = torch.from_numpy(gen.draw_tokens(dims, T, 0, cfg.token_kind)).to(res.dev)
    x = torch.empty((T, dims.hidden), dtype=torch.int16, device=res.dev)
    q.moe_rmsnorm(r, x, stream=stream)
    out = torch.empty((T, dims.hidden), dtype=torch.int16, device=res.dev)
    ws = q.make_workspace(dims, T, res.dev)
    with torch.cuda.stream(stream):
        q.moe_layer_forward(dims, dl, x, out, ws, stream=stream)
        stream.synchronize()
        if q.moe_get_device_status(ws, stream) != q.STRATA_OK:
            raise RuntimeError("prefill: device status")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            q.moe_layer_forward(dims, dl, x, out, ws, stream=stream)
        us = replay_timed([g], reps, args.warmup, stream, ctl, clocks) * 1e3
        prof = None
        acc = {}
        for _ in range(3):
            prof = q.moe_layer_profile(dims, dl, x, out, ws, stream=stream)
            for k, v in prof.items():
                acc[k] = acc.get(k, 0.0) + v / 3
    total, gu_flops = prefill_flops(dims, T)
    _, peak, sustained, src = measured_peaks()
    gu_us = acc["gemm_gate_up"]
    tfl = gu_flops / (gu_us / 1e6) / 1e12
    return {"workload": cfg.description, "tokens": T, "tok_per_s": T * ctl.world / (us / 1e6),
            "us_per_layer": us, "dtype": "f16",
            "arithmetic": "int4 weights dequantised to fp16 x fp16 activations on tcgen05, "
                          "fp32 accumulate",
            "roofline": {"kernel": "k_pf_gemm_sab<gate/up>", "bound": "tensor", "achieved": tfl,
                         "peak": peak, "unit": "TFLOP/s", "frac": tfl / peak,
                         "peak_source": f"{src} bf16 dense (fp16 runs at the same rate), burst",
                         "traffic": kernel_traffic("k_pf_gemm_sab<1>@prefill_T2048"),
                         "us_per_launch": gu_us, "algorithmic_flops_per_launch": gu_flops},
            "tc_frac_whole_layer": total / (us / 1e6) / 1e12 / peak,
            "tc_frac_whole_layer_of_sustained": total / (us / 1e6) / 1e12 / sustained,
            "kernels_us": {k: round(v, 2) for k, v in acc.items()},
            "gpu_launches_per_step": len(prof)}


# --------------------------------------------------------------- oracle leg
def oracle_rate(dims, planes, xs_host, budget_s: float, nthreads: int):
    """Layer-tokens per second of the C oracle: whole layer forwards, layers
    and token variants cycling, until budget_s has passed (at least one)."""
    import oracle
    oracle.build()
    n = tok = 0
    t0 = time.perf_counter()
    while True:
        li = n % len(planes)
        x = xs_host[(n // len(planes)) % len(xs_host)][li]
        oracle.moe_forward(dims, planes[li], x, nthreads=nthreads)
        n += 1
        tok += x.shape[0]
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    return tok / dt, n, dt


def cpu_baseline_block(res, xs_dev, budget):
    xs = [[x.cpu().numpy().view(np.uint16) for x in row] for row in xs_dev[:2]]
    cores = os.cpu_count() or 1
    v1, n1, d1 = oracle_rate(res.dims, res.planes, xs, budget / 2, 1)
    vn, nn, dn = oracle_rate(res.dims, res.planes, xs, budget / 2, cores)
    return {"value": vn, "unit": "tok/s", "cores": cores, "kind": "oracle",
            "single_core": {"value": v1, "unit": "tok/s", "cores": 1},
            "cpu_model": cpu_model(),
            "sample": f"{nn} layer-token forwards at {cores} threads in {dn:.1f} s, {n1} at one "
                      f"thread in {d1:.1f} s (T=1, layers 0..9 and two token variants "
                      "cycling; the C oracle, fp32, OpenMP over experts)"}


def decode1_config(args, world):
    cfg = gen.CONFIGS["decode1"]
    return {"workload": cfg.description, "tokens_per_call": cfg.tokens,
            "layers_per_step": args.layers, "token_variants": args.variants,
            "token_seeds": "1000 * variant + layer",
            "value_unit": "layer-tokens per second (one token through one MoE layer)",
            "l2": f"inputs larger than L2: {args.layers} layers x 455.8 MB resident, "
                  f"{args.variants} token variants per layer rotating between steps",
            "arithmetic": "int4 weights x bf16 activations, fp32 accumulate",
            "parallelism": "replicas" if world > 1 else "single GPU"}


# ------------------------------------------------------------------ runs
def profile_run(q, res, args, stream):
    """Lean run for ncu: the workload's plain calls (no graphs, no stage
    timing, no oracle), warm-up + steps of them, on the resident layers."""
    import torch
    dev, dims = res.dev, res.dims
    if args.workload == "prefill":
        cfg = gen.CONFIGS["prefill"]
        T, kind = cfg.tokens, cfg.token_kind
        layers = [res.layers[0].with_bias(gen.zipf_bias(dims.n_experts, cfg.alpha, 0), dev)]
    elif args.workload == "decode16":
        T, kind = 16, "pairs"
        layers = res.biased(len(res.layers), gen.CONFIGS["decode16"].alpha)
    else:
        T, kind = (args.tokens if args.workload == "stack" else 1), "resid"
        layers = res.layers
    ws = q.make_workspace(dims, T, dev)
    with torch.cuda.stream(stream):
        if args.workload == "stack":
            r0 = torch.from_numpy(gen.draw_tokens(dims, T, 5000, "resid")).to(dev)
            resid = torch.empty_like(r0)
            for _ in range(args.warmup + args.steps):
                resid.copy_(r0)
                q.moe_stack_forward(dims, layers, resid, ws, stream=stream)
        else:
            xs, outs = [], []
            for li in range(len(layers)):
                r = torch.from_numpy(gen.draw_tokens(dims, T, token_seed(0, li), kind)).to(dev)
                x = torch.empty((T, dims.hidden), dtype=torch.int16, device=dev)
                q.moe_rmsnorm(r, x, stream=stream)
                xs.append(x)
                outs.append(torch.empty_like(x))
            for _ in range(args.warmup + args.steps):
                for li in range(len(layers)):
                    q.moe_layer_forward(dims, layers[li], xs[li], outs[li], ws, stream=stream)
        stream.synchronize()
        st = q.moe_get_device_status(ws, stream)
    if st != q.STRATA_OK:
        raise RuntimeError(f"profile run: device status {st}")
    return {"profile": True, "workload": args.workload, "layers": len(layers), "tokens": T}


def run_strata(args, rank, world, local, ctl):
    import torch
    import quantized_moe_expert_fwd_gb300 as q
    q.build.build()
    q.load()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    want_all = args.workload == "decode1" and not args.no_blocks and not args.profile
    n_layers = N_STACK if (want_all or args.workload == "stack") else args.layers
    if args.profile:
        n_layers = args.layers
    res = Resident(dev, n_layers)
    dims = res.dims
    if args.profile:
        return profile_run(q, res, args, stream)
    clocks = ClockSampler(dev).start()
    try:
        if args.workload == "stack":
            blk = stack_block(q, res, args.tokens, args, ctl, clocks, stream, steps=args.steps)
            line = {"metric": METRIC, "value": blk["value"], "unit": "tok/s", "n_gpus": world,
                    "steps": blk["steps"], "warmup": args.warmup,
                    "ms_per_step": blk["ms_per_step"], "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                    "data": "synthetic (seeded random int4 weights and activations of the real "
                            "shapes)",
                    "config": {"workload": f"{gen.CONFIGS['stack'].description}; "
                                           f"T={args.tokens}",
                               "tokens_per_call": args.tokens, "layers_per_step": N_STACK,
                               "value_unit": "tokens per second through the 40-layer stack",
                               "l2": "inputs larger than L2: 18.2 GB of weights resident"},
                    **{k: v for k, v in blk.items() if k not in ("value", "ms_per_step")},
                    "gpu_launches": blk["steps"] * blk["gpu_launches_per_step"],
                    "cpu_baseline": None, "e2e": None, "clocks": clocks.summary()}
            return line
        if args.workload == "prefill":
            pf = prefill_block(q, res, args, ctl, clocks, stream, reps=args.steps)
            return {"metric": METRIC, "value": pf["tok_per_s"], "unit": "tok/s",
                    "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": pf["us_per_layer"] / 1e3, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f16",
                    "data": "synthetic (seeded random int4 weights and activations of the real "
                            "shapes)",
                    "config": {"workload": pf["workload"], "tokens_per_call": pf["tokens"],
                               "value_unit": "prompt tokens per second through one MoE layer",
                               "l2": "inputs larger than L2: 455.8 MB of weights read a step",
                               "arithmetic": pf["arithmetic"]},
                    "roofline": pf["roofline"], "tc_frac_whole_layer": pf["tc_frac_whole_layer"],
                    "kernels_us": pf["kernels_us"],
                    "gpu_launches": args.steps * pf["gpu_launches_per_step"],
                    "cpu_baseline": None, "e2e": None, "clocks": clocks.summary()}
        T, kind, alpha = (1, "resid", None) if args.workload == "decode1" else \
            (16, "pairs", gen.CONFIGS["decode16"].alpha)
        main = decode_block(q, res, T, kind, alpha, args, ctl, clocks, stream,
                            want_e2e=not args.no_e2e)
        xs = main.pop("_xs")
        cfg = decode1_config(args, world) if T == 1 else {
            "workload": gen.CONFIGS["decode16"].description, "tokens_per_call": 16,
            "layers_per_step": args.layers, "value_unit": "layer-tokens per second"}
        line = {"metric": METRIC, "value": main["value"] * world, "unit": "tok/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded random int4 weights and activations of the real "
                        "shapes)",
                "config": cfg, "expert_weight_gbs": main["expert_weight_gbs"],
                "expert_weight_frac_of_8tbs": main["expert_weight_frac_of_8tbs"],
                "touched_experts_per_layer": main["touched_experts_per_layer"],
                "us_per_layer": main["us_per_layer"], "path": main["path"],
                "roofline": main["roofline"], "e2e": main.get("e2e"),
                "gpu_launches": args.steps * main["gpu_launches_per_step"]}
        if want_all and world == 1:
            d16 = decode_block(q, res, 16, "pairs", gen.CONFIGS["decode16"].alpha, args, ctl,
                               clocks, stream)
            d16.pop("_xs")
            line["decode16"] = {"workload": gen.CONFIGS["decode16"].description, **d16}
            for Ts in (1, 4):
                line[f"stack_t{Ts}"] = {"workload": gen.CONFIGS["stack"].description,
                                        **stack_block(q, res, Ts, args, ctl, clocks, stream)}
            line["prefill"] = prefill_block(q, res, args, ctl, clocks, stream)
        line["clocks"] = clocks.summary()
        if rank == 0 and world == 1 and args.cpu_budget > 0 and T == 1:
            line["cpu_baseline"] = cpu_baseline_block(res, xs, args.cpu_budget)
        else:
            line["cpu_baseline"] = None
        return line
    finally:
        clocks.stop()


def run_reference(args, rank, world):
    """The CPU oracle, as it stands, on the host cores: each step one token
    through each of the 10 decode layers, the GPU arm's layers and token
    seeds, bounded so the run ends within a few minutes."""
    import oracle
    oracle.build()
    dims = gen.QWEN
    nl = N_LAYERS
    planes = list(draw_layers(dims, range(nl)))
    nvar = args.variants
    xs = [[oracle.rmsnorm(gen.draw_tokens(dims, 1, token_seed(v, li), "resid"))
           for li in range(nl)] for v in range(nvar)]
    cores = os.cpu_count() or 1

    def step(i):
        v = i % nvar
        for li in range(nl):
            oracle.moe_forward(dims, planes[li], xs[v][li], nthreads=cores)

    t0 = time.perf_counter()
    step(0)
    t_step = time.perf_counter() - t0
    budget = 150.0
    k = args.steps
    if (args.steps + args.warmup) * t_step > budget:
        k = max(3, int(budget / t_step) - args.warmup)
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(k):
        step(i + args.warmup)
    dt = time.perf_counter() - t0
    value = k * nl / dt
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
        "config": decode1_config(args, world),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{k} steps of one token through each of {nl} layers (the "
                                   f"C oracle, fp32, {cores} OpenMP threads) in {dt:.1f} s"},
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
    ap.add_argument("--layers", type=int, default=N_LAYERS,
                    help="decode workloads: distinct layers a step (profile runs: layers resident)")
    ap.add_argument("--profile", action="store_true",
                    help="lean run for ncu: plain calls, no graphs, stage timing, e2e or oracle")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-blocks", action="store_true",
                    help="the decode1 line without its decode16 / stack / prefill blocks")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
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
    try:
        line = run_strata(args, rank, world, local, ctl)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        ctl.close()


if __name__ == "__main__":
    main()
