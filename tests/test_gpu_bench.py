"""The bench's JSON line on a small workload, run with the flags of the benchmark contract.

The tiny workload's inputs fit in L2, so the timed steps must be flushed
(each bracketed by its own events); the line must count our launches and
carry the per-step spread, the roofline and the CPU baseline."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny", "--steps", "20",
           "--warmup", "3", "--e2e-steps", "2", "--cpu-seconds", "0.5", *extra]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])


def test_small_workload_line_is_flushed_and_complete():
    d = _line("--cpu-threads", "1")
    assert d["config"]["l2"].startswith("flushed")
    assert d["gpu_launches"] >= 20
    spread = d["per_step_ms"]
    assert spread["steps"] == 20 and 0 < spread["min"] <= spread["median"]
    # the mean of the flushed steps is the reported time
    assert spread["min"] <= d["ms_per_step"]
    assert d["roofline"]["frac"] > 0 and d["roofline"]["achieved"] > 0
    assert 0 < d["exp_roofline"]["frac"] < 1.5 and d["exp_roofline"]["exps"] == 2 * 256 * 256
    assert d["cpu_baseline"]["cores"] == 1 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0


def test_small_backward_line_is_flushed():
    d = _line("--pass", "backward")
    assert d["config"]["l2"].startswith("flushed")
    assert d["per_step_ms"]["steps"] == 20 and d["value"] > 0


def test_general_entry_point_line_on_strided_cross_shapes():
    d = _line("--layout", "bnhd", "--nk", "300", "--dv", "64", "--cpu-seconds", "0")
    c = d["config"]
    assert c["layout"] == "bnhd" and c["Nk"] == 300 and c["dv"] == 64 and c["Nq"] == 256
    # 2 * B * H * Nq * Nk * (dk + dv) for the tiny workload's B=1, H=2, dk=64
    assert d["roofline"]["algorithmic_flops"] == 2.0 * 1 * 2 * 256 * 300 * (64 + 64)
    assert d["gpu_launches"] >= 20 and d["value"] > 0
