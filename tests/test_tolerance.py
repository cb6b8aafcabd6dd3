"""The parity tolerance's helpers (CPU)."""
import numpy as np
import torch

from tests import gpu_util as G


def test_half_ulp_bounds_bf16_rounding():
    v = np.random.default_rng(0).normal(0, 5, 50000).astype(np.float32)
    r = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    ratio = np.abs(r - v) / G.bf16_half_ulp(v)
    assert ratio.max() <= 1.0 and ratio.max() > 0.99


def test_excess_is_zero_for_a_correct_bf16_rounding_and_catches_errors():
    ref = np.random.default_rng(1).normal(0, 1, (8, 512))
    got = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).float().numpy()
    assert G.excess_stats(got, ref) == 0.0
    bad = got.copy()
    bad[3, 7] += 0.05 * np.sqrt((ref ** 2).mean())
    assert G.excess_stats(bad, ref) > 0.02
