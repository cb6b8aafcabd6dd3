import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size oracle runs (minutes of CPU)")


def pytest_terminal_summary(terminalreporter):
    """The parity figures of every float comparison the GPU tests made: the
    literal max-abs / rms beside the one beyond the bf16 output rounding."""
    try:
        from tests import gpu_util
    except ImportError:
        return
    recs = gpu_util.RECORDS
    if not recs:
        return
    tr = terminalreporter
    lit = [r for r in recs if r[3] > gpu_util.MAX_ABS_RMS]
    tr.write_sep("-", f"parity: {len(recs)} float comparisons")
    tr.write_line(f"worst rel_l2 {max(r[2] for r in recs):.3e} (bar {gpu_util.REL_L2:.0e}); "
                  f"worst literal max_abs/rms {max(r[3] for r in recs):.3e}; worst beyond "
                  f"bf16 rounding {max(r[4] for r in recs):.3e} (bar {gpu_util.MAX_ABS_RMS:.0e})")
    tr.write_line(f"{len(lit)} bf16 comparisons above the literal max-abs bar (within it once "
                  "the output's own rounding is set aside); fp32 comparisons meet it literally")
    for what, dt, rel, mx, ex in sorted(recs, key=lambda r: -r[3])[:8]:
        tr.write_line(f"  {what[:60]:60s} {dt:4s} rel {rel:.2e} literal {mx:.2e} beyond {ex:.2e}")
