"""The bench's multi-rank host logic on CPU (gloo, world size 2).

The forward pass has no exchange step, so N GPUs run independent replicas;
what needs checking is the host side: the max-over-ranks of the timed region,
the whole-job aggregate, and that under torchrun only rank 0 prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        ms = bench.reduce_max(local_ms, dist)
        out[rank] = (ms, bench.aggregate_tflops(1e12, ms, world))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        got = dict(out)
    assert got[0] == got[1]
    ms, tflops = got[0]
    assert ms == 15.0
    assert tflops == pytest.approx(2 * 1e12 / 15e-3 / 1e12)


def test_single_rank_helpers():
    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.aggregate_tflops(2e12, 1.0, 1) == pytest.approx(2000.0)


def test_reference_arm_prints_once_under_torchrun():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_source_digest_ignores_comments_only():
    """The kernel-source digest that ties a profile to the code it was taken
    on leaves comments and blank lines out, keeps string literals whole, and
    changes with the code."""
    a = 'int x = 1; // old note\n/* block */ const char *s = "p//q";\n\nx++;\n'
    b = 'int x = 1; // new note\n\n/* another\n block */ const char *s = "p//q";\nx++;  // more\n'
    c = 'int x = 2; // old note\n/* block */ const char *s = "p//q";\n\nx++;\n'
    assert bench.source_code(a) == bench.source_code(b)
    assert bench.source_code(a) != bench.source_code(c)
    assert '"p//q"' in bench.source_code(a)


def test_l2_plan_flushes_only_inputs_that_fit():
    l2 = 129 << 20
    nbytes, text = bench.l2_plan(l2, 403 << 20)
    assert nbytes == 0 and text.startswith("no flush")
    nbytes, text = bench.l2_plan(l2, 264 * 1024)
    assert nbytes == 2 * l2 and text.startswith("flushed")
    # an input exactly the size of L2 still fits in it
    assert bench.l2_plan(l2, l2)[0] == 2 * l2


def test_reference_arm_honours_the_thread_count():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "1", "--warmup", "3", "--cpu-threads", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert d["cpu_baseline"]["cores"] == 1


def test_attention_counts_match_brute_force():
    # pairs the mask keeps, counted one by one on a small ragged shape
    B, H, Nq, Nk, dk, dv = 2, 3, 7, 5, 16, 8
    for causal in (False, True):
        pairs = sum(1 for i in range(Nq) for j in range(Nk) if not causal or j <= i)
        flops, nbytes = bench.attention_counts(B, H, Nq, Nk, dk, dv, causal, 2)
        assert flops == 2.0 * B * H * pairs * (dk + dv)
        assert nbytes == B * H * (2 * (Nq * dk + Nk * dk + Nk * dv + Nq * dv) + 4 * Nq)
    # the self-attention bench counts: 4 B H N^2 d unmasked
    f, _ = bench.attention_counts(4, 32, 4096, 4096, 128, 128, False, 2)
    assert f == 4.0 * 4 * 32 * 4096 ** 2 * 128


def test_step_spread_reports_min_and_median():
    s = bench.step_spread([0.5, 0.6, 0.7, 0.9])
    assert s["min"] == 0.5 and s["steps"] == 4 and s["median"] == pytest.approx(0.65)


def test_exp_roofline_counts_the_kept_pairs():
    """One exponential per (query, key) pair the mask keeps: N^2 per head, or
    N (N + 1) / 2 with the causal mask, against 32 per clock per SM."""
    import synth
    w = synth.Workload("t", 2, 3, 5, 64, "bf16", False, seed=1)
    r = bench.exp_roofline(w, 1.0, 152, 2000)
    assert r["exps"] == 2 * 3 * 25
    assert r["peak"] == pytest.approx(32 * 152 * 2000e6 / 1e12)
    assert r["achieved"] == pytest.approx(150 / 1e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    wc = synth.Workload("t", 2, 3, 5, 64, "bf16", True, seed=1)
    assert bench.exp_roofline(wc, 1.0, 152, None)["exps"] == 2 * 3 * 15


def test_traffic_only_for_the_named_workload():
    """A resized workload (--batch, --heads, --seq) gets no ncu traffic figure:
    the committed summaries hold the named workload's bytes per launch."""
    import synth
    w = synth.WORKLOADS["multihead"]
    assert bench.traffic_for("tc", w) == bench.profiled_traffic("tc", "multihead")
    for small in (w.scaled(B=1), w.scaled(H=64), w.scaled(N=1024)):
        traffic, note = bench.traffic_for("tc", small)
        assert traffic is None and "resized" in note
