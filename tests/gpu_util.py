"""Helpers of the GPU parity tests: device upload, the tolerance, the
near-tie rule.

Tolerance of floating outputs (bf16 from the GPU against the fp32 oracle):
relative L2 <= 5e-3 and max |diff| <= 2e-2 * rms(reference).
Near ties: a token whose oracle K-th and (K+1)-th logits differ by less than
1e-4 may be routed differently by an fp32 sum taken in another order; its ids
are not compared, and its floats are checked on a run with the oracle's
routing forced.
"""
import numpy as np
import torch

REL_L2 = 5e-3
MAX_ABS_RMS = 2e-2
NEAR_TIE = 1e-4


def dev():
    return torch.device("cuda:0")


def u16(a, device=None):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device or dev())


def f32(a, device=None):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device or dev())


def i32(a, device=None):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device or dev())


def bf16_to_np(t):
    return t.view(torch.bfloat16).float().cpu().numpy()


def err_stats(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    rms = float(np.sqrt((want ** 2).mean())) if want.size else 0.0
    rel = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    mx = float(np.abs(got - want).max() / max(rms, 1e-30)) if want.size else 0.0
    return rel, mx


def assert_close(got, want, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel, mx = err_stats(got, want)
    assert rel <= REL_L2 and mx <= MAX_ABS_RMS, f"{what}: rel_l2 {rel:.3e}, max_abs/rms {mx:.3e}"
    return rel, mx


def clear_tokens(gap):
    return [t for t in range(len(gap)) if not (gap[t] < NEAR_TIE)]
