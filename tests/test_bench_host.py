"""Host-side pieces of bench.py (no GPU): argument defaults, the byte model, the traffic record,
the clock-sample parser."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_defaults_run_the_full_scale_workload():
    a = bench.parse_args([])
    assert a.cfg == 3 and a.gpus == 1 and a.warmup >= 3 and a.impl == "ours"


def test_algorithmic_bytes_per_token():
    lay = synth.make_layout("full", 1)
    assert bench.algo_bytes_per_token(lay) == 18_624  # 2 x 24 x (128 + 4 + 256)
    assert bench.algo_bytes_per_token(synth.make_layout("tiny", 1)) == 6 * (32 + 4 + 64)


def test_traffic_record_matches_the_kernel_sources():
    # the committed ncu record is only used for the kernel it was taken on
    t = bench.recorded_traffic(3)
    assert t is None or 1.2e9 < t < 2.0e9
    assert bench.recorded_traffic(1) is None


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1900, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active"]
    s = c.summary()
    assert s["sm_mhz"] == 1985 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
