"""Where the persistent kernel's time goes, phase by phase.

Builds the phase-traced library (build.build(trace=True): the same sources
compiled with STRATA_PX_TRACE, a separate .so), runs the one-token layer of
the 2048-hidden, 256-expert, top-8 shape as the decode benchmark does (10
distinct layers in a CUDA graph, 16 token variants rotating) and the
40-layer stack, and prints the medians over the CTAs of every phase point of
the last launch (global-timer stamps; the stores cost about a microsecond a
layer against the untraced build).

    python -m quantized_moe_expert_fwd_gb300.phase_trace [--steps N]
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

from . import build as _build
from . import strata_moe as q

POINTS = ["CTA initialised", "dependency resolved", "token row in smem", "router + shared pairs",
          "logits seen", "top-K + gate", "plan published", "gate/up done", "SwiGLU staged",
          "down done", "combined", "producer: plan seen", "producer: gate/up issued",
          "producer: down issued"]


def _medians(rec, slot, ref):
    """Median over the CTAs of each point of `slot`, µs after point `ref`
    of the same slot (points never written: nan)."""
    s = rec[:, slot, :len(POINTS)].astype(np.float64)
    s[s == 0] = np.nan
    med = np.array([np.median(c[~np.isnan(c)]) if (~np.isnan(c)).any() else np.nan
                    for c in s.T])
    return (med - med[ref]) / 1000.0


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--steps", type=int, default=300, help="graph replays before the record")
    args = ap.parse_args(argv)
    q.use_library(_build.build(trace=True))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    from workloads import gen
    dev = torch.device("cuda:0")
    dims, nl, nv = gen.QWEN, 10, 16
    G = torch.cuda.get_device_properties(dev).multi_processor_count
    layers = [q.DeviceLayer(gen.draw_layer(dims, s), dev) for s in range(nl)]
    xs = []
    for v in range(nv):
        row = []
        for li in range(nl):
            r = torch.from_numpy(gen.draw_tokens(dims, 1, 1000 * v + li, "resid")).to(dev)
            x = torch.empty((1, dims.hidden), dtype=torch.int16, device=dev)
            q.moe_rmsnorm(r, x)
            row.append(x)
        xs.append(row)
    outs = [torch.empty((1, dims.hidden), dtype=torch.int16, device=dev) for _ in range(nl)]
    ws = q.make_workspace(dims, 1, dev)
    st = torch.cuda.Stream(dev)
    with torch.cuda.stream(st):
        graphs = []
        for v in range(nv):
            for li in range(nl):
                q.moe_layer_forward(dims, layers[li], xs[v][li], outs[li], ws, stream=st)
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for li in range(nl):
                    q.moe_layer_forward(dims, layers[li], xs[v][li], outs[li], ws, stream=st)
            graphs.append(g)
        for i in range(args.steps):
            graphs[i % nv].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for i in range(args.steps):
            graphs[i % nv].replay()
        e1.record(st)
        e1.synchronize()
        per_layer = e0.elapsed_time(e1) * 1e3 / (args.steps * nl)
        if q.moe_get_device_status(ws, st) != 0:
            raise RuntimeError("device status after the one-layer runs")
    one = q.strata_px_trace_read()[:G]
    r0 = torch.from_numpy(gen.draw_tokens(dims, 1, 77, "resid")).to(dev)
    resid = torch.empty_like(r0)
    with torch.cuda.stream(st):
        for _ in range(5):
            resid.copy_(r0)
            q.moe_stack_forward(dims, layers * 4, resid, ws, eps=1e-6, stream=st)
        st.synchronize()
        if q.moe_get_device_status(ws, st) != 0:
            raise RuntimeError("device status after the stack runs")
    stack = q.strata_px_trace_read()[:G]

    print(f"one-token layer, traced build: {per_layer:.2f} us a layer in the graph of {nl} layers")
    print("  medians over the CTAs of the last launch, us after the grid dependency resolved:")
    m = _medians(one, 0, 1)
    for i, name in enumerate(POINTS):
        print(f"    {i:2d} {name:26s} {m[i]:7.2f}")
    print("40-layer stack (one launch): medians over the CTAs, us after the layer's token row:")
    print(f"    {'':29s}" + "".join(f"{h:>10s}" for h in ("layer 0", "layer 1", "layer 20", "layer 39")))
    cols = [_medians(stack, s, 2) for s in range(4)]
    for i, name in enumerate(POINTS):
        if i < 2:
            continue
        print(f"    {i:2d} {name:26s}" + "".join(f"{c[i]:10.2f}" for c in cols))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
