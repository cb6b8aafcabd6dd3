"""Host-side pieces of bench.py: the clock record kept for the timed windows,
the per-launch DRAM traffic looked up against the kernel source's digest,
and the CPU description of the oracle's timing."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler(samples, windows, max_mhz=2070.0):
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.samples, c.windows, c.max_mhz, c.error = samples, windows, max_mhz, None
    return c


def test_clock_summary_keeps_only_timed_windows():
    samples = [(0.5, 900.0, 0x1), (1.1, 1950.0, 0x4), (1.2, 1965.0, 0x0),
               (1.3, 1980.0, 0x4), (3.0, 600.0, 0x8 | 0x40)]
    s = _sampler(samples, [(1.0, 1.5)]).summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1965.0
    assert s["sm_max_mhz"] == 2070.0
    # idle (0x1) and the slow-down outside the window are not reported
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_decodes_every_named_reason():
    bits = 0x4 | 0x8 | 0x20 | 0x40 | 0x80
    s = _sampler([(1.0, 1000.0, bits)], [(0.0, 2.0)]).summary()
    assert s["reasons"] == sorted(["sw_power_cap", "hw_slowdown", "sw_thermal_slowdown",
                                   "hw_thermal_slowdown", "hw_power_brake_slowdown"])


def test_clock_summary_without_nvml_says_so():
    c = _sampler([], [])
    c.error = "no library"
    s = c.summary()
    assert s["sm_mhz"] is None and s["reasons"] == ["nvml unavailable"]


def test_kernel_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    csrc = tmp_path / "quantized_moe_expert_fwd_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_bytes(b"kernel one")
    (tmp_path / "profiles").mkdir()
    entry = {"source": "k.cu", "sha256": hashlib.sha256(b"kernel one").hexdigest(),
             "bytes_per_launch": 1234}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"k": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k") == 1234
    assert bench.kernel_traffic("other") is None
    (csrc / "k.cu").write_bytes(b"kernel two")
    assert bench.kernel_traffic("k") is None


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        j = json.load(f)
    for name, ent in j.items():
        assert os.path.exists(os.path.join(ROOT, "quantized_moe_expert_fwd_gb300", "csrc",
                                           ent["source"])), name
        assert ent["bytes_per_launch"] > 0
        assert os.path.exists(os.path.join(ROOT, ent["from"])), name


def test_cpu_model_is_named():
    assert bench.cpu_model().strip()


def test_layer_byte_counts():
    d = bench.gen.QWEN
    # one expert: gate+up 2*512 rows of 2048 int4 + fp16 scales per 32,
    # down 2048 rows of 512 int4 + scales
    assert bench.expert_bytes(d) == 1024 * 1024 + 1024 * 64 * 2 + 2048 * 256 + 2048 * 16 * 2
    assert bench.gu_bytes(d, d.inter) + 2048 * 256 + 2048 * 16 * 2 == bench.expert_bytes(d)
    assert bench.router_bytes(d) == 257 * 2048 * 2
    assert bench.token_seed(3, 7) == 3007
