"""Tolerance study of the emulated MXFP8 expert path (oracle/w4a8.py)
against the exact oracle, on the Qwen3.6-35B-A3B layer shape with the
oracle's own routing.  Calls only the oracle and the input generator; prints
one line per case.  Usage: python -m oracle.w4a8_study [T] [n_seeds]"""
from __future__ import annotations

import sys
import time

import numpy as np

import oracle
from oracle import w4a8
from workloads import gen


def main(T: int = 16, n_seeds: int = 3) -> None:
    dims = gen.QWEN
    for seed in range(n_seeds):
        planes = gen.draw_layer(dims, 40 + seed)
        xb = oracle.rmsnorm(gen.draw_tokens(dims, T, 40 + seed, "resid"))
        t0 = time.time()
        ref = oracle.moe_forward(dims, planes, xb)
        ex = w4a8.layer_forward(dims, planes, xb, ref["ids"], ref["w"], ref["sig"], False)
        qz = w4a8.layer_forward(dims, planes, xb, ref["ids"], ref["w"], ref["sig"], True)
        rms = float(np.sqrt(np.mean(ref["out"].astype(np.float64) ** 2)))
        rel = lambda a: float(np.linalg.norm(a - ref["out"]) / np.linalg.norm(ref["out"]))
        print(f"seed {40 + seed} T={T}: harness rel-L2 {rel(ex):.2e}; MXFP8 rel-L2 {rel(qz):.4f}, "
              f"max-abs {np.abs(qz - ref['out']).max() / rms:.3f} rms ({time.time() - t0:.0f} s)",
              flush=True)


if __name__ == "__main__":
    args = [int(a) for a in sys.argv[1:]]
    main(*args)
