"""The bench contract on the host: the reference arm (the float64 oracle) prints one JSON
line with the contract's keys, and the native arm refuses to run without a GPU instead of
falling back to anything on the CPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--workload", "random_dfa_S64_L128"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["warmup"] == 3 and d["steps"] == 2
    assert d["config"]["workload"] == "random_dfa_S64_L128"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    assert cb["cpu_model"]
    assert d["config"]["sequences_per_step"] == 1
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_native_arm_needs_a_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = subprocess.run([sys.executable, "bench.py", "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode != 0
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_default_workload_is_the_block_wise_batch():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.DEFAULT_WORKLOAD == "blockwise_dfa_S512_L512"


def test_clock_summary_keeps_the_timed_window():
    """Samples before mark_start() or after the period following mark_end() are not in the
    summary; throttle reasons seen inside the window are reported."""
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.t0, c.t1 = 10.0, 12.0
    row = "0, %d, 2070, 900.5, 0x0, %s, Not Active, Not Active, %s"
    c.lines = [(9.0, row % (1200, "Active", "Not Active")),        # before the window: ignored
               (10.5, row % (2000, "Not Active", "Not Active")),
               (11.5, row % (2010, "Not Active", "Active")),
               (12.1, row % (1990, "Not Active", "Not Active")),   # within one period after the end
               (13.0, row % (500, "Active", "Not Active"))]         # long after: ignored
    s = c.summary()
    assert s["samples_in_timed_region"] == 3 and s["samples"] == 3
    assert s["sm_mhz"] == 2000.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
