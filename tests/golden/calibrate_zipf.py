"""Choose the Zipf(s=1.1) router-bias strength alpha of the skewed workloads.

Routes synthetic Qwen-shaped tokens through the oracle (router logits once,
then top-K selection for each candidate bias) and prints, per alpha:
  share20  the fraction of all selections that land on the 20% most selected
           experts (the decode T=16 workload wants about 0.80)
  min/max  the smallest and largest expert load at T=2048 (the prefill
           workload wants about 10 and about 300)
Calls only the oracle and the input generator.  Usage:
  python tests/golden/calibrate_zipf.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle  # noqa: E402
from workloads import gen  # noqa: E402


def share_top20(ids, E):
    c = np.sort(np.bincount(ids.ravel(), minlength=E))[::-1]
    return c[: int(round(0.2 * E))].sum() / c.sum()


def main():
    dims = gen.QWEN
    E, K = dims.n_experts, dims.top_k
    L = gen.draw_layer(dims, 0)
    r = gen.draw_tokens(dims, 4096, 123, "resid")
    x = oracle.rmsnorm(r)
    logits, _ = oracle.router(x, L["router"], None)
    rp = gen.draw_tokens(dims, 2048, 0, "resid")
    lp, _ = oracle.router(oracle.rmsnorm(rp), L["router"], None)
    for alpha in np.arange(0.4, 2.01, 0.1):
        b = gen.zipf_bias(E, alpha, 0)
        ids, _, _ = oracle.select(logits + b, K)
        idp, _, _ = oracle.select(lp + b, K)
        loads = np.bincount(idp.ravel(), minlength=E)
        print(f"alpha {alpha:.2f}  share20 {share_top20(ids, E):.3f}  "
              f"prefill loads min {loads.min()} max {loads.max()}")


if __name__ == "__main__":
    main()
