"""bench.py on a GPU, reduced long-context batch: the JSON line's roofline is
a per-call mean over at least 200 back-to-back decode calls, no longer than
a whole step, and consistent with the step rate; the clocks and the e2e leg
are present."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_is_consistent(cuda_device):
    cmd = [sys.executable, "bench.py", "--workload", "long", "--num-seqs", "1",
           "--num-blocks", "4096", "--steps", "10", "--warmup", "3", "--no-cpu-baseline"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    roof = line["roofline"]
    assert roof["timed_launches"] >= 200 and roof["sampled_calls"] >= 20
    assert roof["per_call_le_step"] is True
    assert roof["decode_ms_mean"] <= line["ms_per_step"] * 1.02
    # the call's rate and the step's rate agree within the write and ramp-up
    step_rate = line["bytes_per_step"]["decode"] / (line["ms_per_step"] / 1e3) / 1e9
    assert 0.9 * step_rate <= roof["achieved"] <= 1.25 * step_rate
    assert roof["clocks"]["samples"] >= 1 and line["clocks"]["samples"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["e2e"]["d2h_bytes_per_step"] > 0
    assert line["gpu_launches"] >= 2 * line["steps"]
    assert line["config"]["num_seqs"] == 1 and line["config"]["name"] == "long"
