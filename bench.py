"""Benchmark of the attention forward pass on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload multihead|causal|peaked|tiny|large_d]
                  [--batch B] [--heads H] [--seq N] [--pass forward|backward]
                  [--layout bhnd|bnhd] [--nk NK] [--dv DV]

One step = one forward pass (fa_forward, one kernel launch) over the whole
workload.  Default workload: B=4, H=32, N=4096, d=128, bf16, non-causal --
the multi-head shape the throughput target is quoted on.  Inputs are the
seeded synthetic tensors of ``synth`` (i.i.d. N(0,1), rounded to bf16),
resident in HBM before timing.  Q, K and V (403 MB) are larger than L2
(129 MB), so no flush is needed between steps; workloads whose inputs fit in
L2 (tiny, large_d) write a buffer of twice L2 before each timed step, each
step bracketed by its own events.

Prints one JSON line (rank 0).  ``value`` is TFLOP/s = 4*B*H*N^2*d / time
(halved under a causal mask) summed over ranks; ``e2e`` is the same metric
through fa_forward_host with pinned host buffers, the copies inside the
timed region; ``roofline`` relates the kernel to the measured bf16 tensor
peak; ``cpu_baseline`` times the CPU oracle on a bounded row sample.

``--impl reference`` times that oracle (the plain CPU definition) as the
reference arm on the same workload, a bounded row sample per step.
Under torchrun (N > 1) every rank runs the whole workload on its own GPU
(independent replicas: the forward pass has no exchange step).

``--layout``, ``--nk`` or ``--dv`` time the general entry point fa_attention
instead: strided (batch, seq, heads, dim) storage, key counts other than the
query count, value widths other than d; ``--pass backward`` times fa_backward.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "attention fwd TFLOP/s (4·B·H·N²·d/time) and % of GB300 BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {"tc": "tiled_online_softmax_attn_gb300/csrc/fa_tc.cu",
                  "wide": "tiled_online_softmax_attn_gb300/csrc/fa_wide.cu",
                  "general": "tiled_online_softmax_attn_gb300/csrc/fa_general.cu"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(w):
    return (f"{w.name}: B={w.B} H={w.H} N={w.N} d={w.d} {w.dtype}"
            f"{' causal' if w.causal else ''}{' QK x%g' % w.qk_mult if w.qk_mult != 1 else ''}")


def source_code(text):
    """The source without comments and blank lines, so that a comment edit
    does not count as a change of the kernel (string literals kept as they are)."""
    out, i, n, quote = [], 0, len(text), None
    while i < n:
        c = text[i]
        if quote:
            out.append(c)
            if c == "\\" and i + 1 < n:
                out.append(text[i + 1])
                i += 2
                continue
            if c == quote:
                quote = None
            i += 1
        elif c in "\"'":
            quote = c
            out.append(c)
            i += 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def source_digest(path):
    """sha256 prefix of a kernel source's code (comments and blank lines left out)."""
    with open(os.path.join(ROOT, path), encoding="utf-8") as f:
        return hashlib.sha256(source_code(f.read()).encode()).hexdigest()[:16]


def profiled_traffic(kernel_key, workload):
    """(DRAM bytes per launch, how they were counted) from a committed ncu
    summary, if it was taken on the current kernel source (matching digest)
    for this workload; (None, reason) otherwise."""
    path = os.path.join(ROOT, "profiles", f"ncu_{kernel_key}_{workload}.md")
    if not os.path.exists(path):
        return None, "no ncu summary for this kernel and workload"
    text = open(path).read()
    m_d = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    m_t = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    m_n = re.search(r"traffic_note:\s*(.+)", text)
    if not m_d or not m_t:
        return None, "the ncu summary holds no traffic figure"
    if m_d.group(1) != source_digest(KERNEL_SOURCES[kernel_key]):
        return None, "the kernel source changed since the ncu capture"
    return float(m_t.group(1)), (m_n.group(1).strip() if m_n else "ncu dram__bytes_read.sum + dram__bytes_write.sum")


def traffic_for(kernel_key, w):
    """profiled_traffic for a workload as named; a resized one (--batch,
    --heads, --seq) has no figure, since the summaries hold the named
    workload's traffic."""
    if w != synth.WORKLOADS.get(w.name):
        return None, "workload resized from the named one: no ncu figure for it"
    return profiled_traffic(kernel_key, w.name)


class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes; no
    Python NVML package needed): SM clock, its maximum, power and the
    active clock-event reasons of one device."""
    SM = 1                                   # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for device %d" % index)
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _uint(self, fn, *args):
        v = self.c.c_uint()
        return v.value if fn(self.h, *args, self.c.byref(v)) == 0 else None

    def sample(self):
        mask = self.c.c_ulonglong()
        ok = self.reasons_fn(self.h, self.c.byref(mask)) == 0
        return (self._uint(self.lib.nvmlDeviceGetClockInfo, self.c.c_uint(self.SM)),
                self._uint(self.lib.nvmlDeviceGetPowerUsage),
                [n for b, n in self.REASONS.items() if ok and mask.value & b])

    def max_sm(self):
        return self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.c.c_uint(self.SM))

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock and clock-event reasons sampled every 2 ms while the timed
    region runs (NVML through ctypes; nvidia-smi every 100 ms where NVML
    cannot be loaded).  Call ``mark_start()`` / ``mark_end()`` around the
    timed region: samples taken between the two count as under load, so a
    timed region of a dozen milliseconds still has its own clock record."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.002

    def __init__(self, gpu_index):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        self.gpu = int(ids[gpu_index]) if gpu_index < len(ids) and ids[gpu_index].isdigit() else gpu_index
        self.proc = None
        self.nvml = None
        self.samples = []          # (time, sm MHz, power mW, reasons)
        self.window = [None, None]
        self.lines = []

    def __enter__(self):
        import threading
        try:
            self.nvml = _Nvml(self.gpu)
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        else:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
        time.sleep(0.05)
        return self

    def _run(self):
        while not self.stop.is_set():
            t = time.perf_counter()
            try:
                clk, pw, why = self.nvml.sample()
            except OSError:
                break
            self.samples.append((t, clk, pw, why))
            self.stop.wait(self.PERIOD_S)

    def mark_start(self):
        self.window[0] = time.perf_counter()

    def mark_end(self):
        self.window[1] = time.perf_counter()

    def __exit__(self, *exc):
        if self.nvml is not None:
            time.sleep(0.01)
            self.stop.set()
            self.thread.join(timeout=5)
            self.max_mhz = self.nvml.max_sm()
            self.nvml.close()
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        if self.nvml is not None:
            t0, t1 = self.window
            load = [s for s in self.samples if t0 is not None and t1 is not None and t0 <= s[0] <= t1]
            sm = [s[1] for s in load if s[1] is not None]
            reasons = sorted({r for s in load for r in s[3]})
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples_under_load": len(sm), "samples": len(self.samples),
                    "source": "NVML every %d ms, samples inside the timed region" % round(self.PERIOD_S * 1e3)}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                clk, mxc, pw = float(f[1]), float(f[2]), float(f[3])
            except ValueError:
                continue
            mx = mxc
            if pw > 200.0:   # samples under load
                sm.append(clk)
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples_under_load": len(sm), "samples": len(self.lines),
                "source": "nvidia-smi every 100 ms, samples above 200 W"}


def oracle_rows_rate(w, q, k, v, seconds, seed=0, threads=0):
    """Times the CPU oracle on a seeded row sample sized for about `seconds`
    on `threads` host threads (0: all of them); returns (TFLOP/s, rows,
    threads, elapsed)."""
    import oracle
    threads = threads or oracle.default_threads()
    rng = np.random.default_rng(seed)
    total = w.B * w.H * w.N
    # rows are drawn with replacement, so a workload smaller than the sample
    # is simply covered several times; the fp64 outputs of one call are kept
    # to about 256 MB
    chunk = max(threads, (32 << 20) // v.shape[-1])
    # calibrate on a growing sample until it runs long enough to be representative
    n_cal = max(threads, 8)
    while True:
        calib = rng.integers(0, total, size=n_cal)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, w.scale, w.causal, calib, threads)
        dt = max(time.perf_counter() - t0, 1e-6)
        if dt >= min(0.5, seconds / 4) or n_cal >= chunk:
            break
        n_cal = min(chunk, n_cal * 4)
    nrows = int(max(threads, n_cal * seconds / dt))
    rows = rng.integers(0, total, size=nrows)
    t0 = time.perf_counter()
    for c in range(0, nrows, chunk):
        oracle.attention_rows(q, k, v, w.scale, w.causal, rows[c:c + chunk], threads)
    el = time.perf_counter() - t0
    i = rows % w.N
    keys = (i + 1) if w.causal else np.full(nrows, w.N)
    flops = float(4.0 * w.d * keys.sum())
    return flops / el / 1e12, nrows, threads, el


def reference_arm(args, w, q, k, v, rank, world):
    """The oracle (plain fp64 CPU definition) timed as the reference arm."""
    if rank != 0:
        return
    per_step = max(0.5, min(10.0, 90.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_rows_rate(w, q, k, v, per_step, seed=1, threads=args.cpu_threads)
    rates, rows_total, el_total, threads = [], 0, 0.0, 1
    for s in range(args.steps):
        r, nrows, threads, el = oracle_rows_rate(w, q, k, v, per_step, seed=100 + s,
                                                 threads=args.cpu_threads)
        rates.append(r)
        rows_total += nrows
        el_total += el
    value = statistics.mean(rates)
    step_flops_full = w.flops
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_flops_full / (value * 1e12) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_desc(w), "B": w.B, "H": w.H, "N": w.N,
                                         "d": w.d, "causal": w.causal, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_total} seeded query rows (full key range each) over "
                                   f"{args.steps} steps, {el_total:.1f} s; ms_per_step extrapolates "
                                   f"to the whole workload"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_e2e(args, w, fa, torch, dev, stream, q_h, k_h, v_h, q, o, lse, tdt, dist, world):
    """The workload end to end through fa_forward_host: host-to-device copy of
    Q, K, V from pinned host memory, the kernels, and the copy of O and LSE
    back, every step inside the timed region."""
    o_h = torch.empty(w.shape, dtype=tdt).pin_memory()
    lse_h = torch.empty(w.shape[:3], dtype=torch.float32).pin_memory()
    ws_bytes = fa.host_workspace_size(w.B, w.H, w.N, w.d, q.dtype, q.dtype)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def e2e_step():
        fa.forward_host(q_h, k_h, v_h, o_h, lse_h, ws, scale=w.scale, causal=w.causal, stream=stream)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps
    e2e_ms = reduce_max(e2e_ms, dist, dev)
    h2d = 3 * q.numel() * q.element_size()
    d2h = o.numel() * o.element_size() + lse.numel() * 4
    # the host-buffer result must be the device result
    if not torch.equal(o_h, o.cpu()) or not torch.equal(lse_h, lse.cpu()):
        raise RuntimeError("host-buffer path disagrees with the device path")
    return {"value": aggregate_tflops(w.flops, e2e_ms, world), "unit": "TFLOP/s",
            "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "fa_forward_host (pinned host buffers, wall clock per synchronous call)"}


def reduce_max(x: float, dist, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job throughput: every rank runs the full workload (replicas), the
    job takes as long as its slowest rank."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def l2_plan(l2_bytes: int, input_bytes: int):
    """How the timed steps keep L2 honest: inputs larger than L2 need nothing
    (each step streams them from HBM again); smaller ones get a buffer of twice
    L2 written before every timed step.  Returns (flush buffer bytes or 0, the
    config text saying which)."""
    if input_bytes > l2_bytes:
        return 0, "no flush: inputs (%.1f MB) exceed L2 (%.0f MB)" % (input_bytes / 1e6, l2_bytes / 1e6)
    return 2 * l2_bytes, ("flushed: a %.0f MB buffer written before each timed step, outside its "
                          "events (inputs %.1f MB fit in L2 %.0f MB)" % (2 * l2_bytes / 1e6, input_bytes / 1e6,
                                                                        l2_bytes / 1e6))


def device_l2_bytes(torch, dev) -> int:
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)


def time_steps(torch, dev, stream, step, steps, flush):
    """Device time of `steps` calls of `step` on `stream`.  Without a flush
    buffer the calls run back to back with an event at every boundary (the
    total is first to last event); with one, each call has its own event pair
    and the buffer is written before it, outside the pair.  Returns (total ms,
    sorted per-step ms)."""
    if flush is None:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record(stream)
        for i in range(steps):
            step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        return evs[0].elapsed_time(evs[-1]), sorted(a.elapsed_time(b) for a, b in zip(evs, evs[1:]))
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in pairs:
            flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
    torch.cuda.synchronize(dev)
    per = sorted(a.elapsed_time(b) for a, b in pairs)
    return sum(per), per


EX2_PER_CLOCK_PER_SM = 32  # GB300's exponential units (twice B200's 16)


def exp_roofline(w, ms_step, sms, sm_max_mhz):
    """The exponential unit's roofline, reported beside the tensor one: one
    ex2 per (query, key) pair the mask keeps, against EX2_PER_CLOCK_PER_SM
    x SMs x the maximum SM clock."""
    pairs = w.B * w.H * (w.N * (w.N + 1) / 2 if w.causal else float(w.N) ** 2)
    mhz = sm_max_mhz or 2070
    peak = EX2_PER_CLOCK_PER_SM * sms * mhz * 1e6 / 1e12
    achieved = pairs / (ms_step * 1e-3) / 1e12
    return {"exps": pairs, "achieved": achieved, "peak": peak, "unit": "Tex2/s", "frac": achieved / peak,
            "peak_source": f"derived: {EX2_PER_CLOCK_PER_SM} ex2 per clock per SM x {sms} SMs x {mhz} MHz"}


def step_spread(per):
    """Minimum and median of the timed region's single steps."""
    return {"min": per[0], "median": statistics.median(per), "steps": len(per)}


def attention_counts(B, H, Nq, Nk, dk, dv, causal, elt):
    """(FLOPs, bytes) of one pass of the general entry point: two products of
    2 d per (query, key) pair that the mask keeps (key <= query when causal),
    Q, K, V read and O, LSE written once."""
    if causal:
        i = np.arange(Nq, dtype=np.float64)
        pairs = float(np.minimum(i + 1, Nk).sum())
    else:
        pairs = float(Nq) * Nk
    flops = 2.0 * B * H * pairs * (dk + dv)
    nbytes = B * H * (elt * (Nq * dk + Nk * dk + Nk * dv + Nq * dv) + 4.0 * Nq)
    return flops, nbytes


def bench_attention(args, w, world, rank, local_rank):
    """fa_attention (the strided, cross-shape entry point) on the workload with
    Nk keys, value width dv and the chosen storage: "bhnd" is contiguous
    [B, H, N, d], "bnhd" is (batch, seq, heads, dim) storage seen through a
    transposed view, for Q, K, V and O alike.  One step = one call."""
    import torch
    import tiled_online_softmax_attn_gb300 as fa
    from tiled_online_softmax_attn_gb300 import build as fa_build
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa_build.build()
    B, H, Nq, dk = w.B, w.H, w.N, w.d
    Nk, dv = args.nk or w.N, args.dv or w.d
    s = w.seed
    q_np = synth.tensor(3 * s, (B, H, Nq, dk), w.dtype, w.qk_mult)
    k_np = synth.tensor(3 * s + 1, (B, H, Nk, dk), w.dtype, w.qk_mult)
    v_np = synth.tensor(3 * s + 2, (B, H, Nk, dv), w.dtype)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def place(x):
        t = torch.from_numpy(x).to(tdt)
        if args.layout == "bhnd":
            return t.to(dev)
        return t.transpose(1, 2).contiguous().to(dev).transpose(1, 2)

    q, k, v = place(q_np), place(k_np), place(v_np)
    o = place(np.zeros((B, H, Nq, dv), dtype=np.float32))
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    ws_bytes = fa.attention_workspace_size(q, k, v, o=o, causal=w.causal)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    per_call = 2 if ws_bytes else 1  # the key-range split adds its combine launch
    stream = torch.cuda.current_stream(dev)
    launches = {"n": 0}

    def step():
        fa.fa_attention(q, k, v, o=o, lse=lse, scale=1.0 / math.sqrt(dk), causal=w.causal,
                        workspace=ws, stream=stream)
        launches["n"] += per_call

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.check_device_error(stream.cuda_stream) != fa.FA_OK:
        raise RuntimeError(fa.last_error())
    elt = 2 if w.dtype == "bf16" else 4
    flops, nbytes = attention_counts(B, H, Nq, Nk, dk, dv, w.causal, elt)
    in_bytes = elt * B * H * (Nq * dk + Nk * dk + Nk * dv)
    flush_bytes, l2_text = l2_plan(device_l2_bytes(torch, dev), in_bytes)
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device=dev) if flush_bytes else None
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches["n"] = 0
    with ClockSampler(local_rank) as clocks:
        clocks.mark_start()
        ms_total, per = time_steps(torch, dev, stream, step, args.steps, flush)
        clocks.mark_end()
    if fa.check_device_error(stream.cuda_stream) != fa.FA_OK:
        raise RuntimeError(fa.last_error())
    ms = reduce_max(ms_total, dist, dev) / args.steps
    value = world * flops / (ms * 1e-3) / 1e12
    peaks, peak_kind = load_peaks()
    t_tensor = flops / (float(peaks["bf16_tflops"]) * 1e12)
    t_hbm = nbytes / (float(peaks["hbm_gbs"]) * 1e9)
    if t_tensor >= t_hbm:
        peak = float(peaks["bf16_tflops"])
        achieved = flops / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak}
    else:
        peak = float(peaks["hbm_gbs"])
        achieved = nbytes / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak}
    roof.update({"peak_source": peak_kind, "traffic": None, "algorithmic_bytes": nbytes,
                 "algorithmic_flops": flops, "launches_per_step": per_call})
    line = {
        "metric": "attention fwd TFLOP/s (2·B·H·Nq·Nk·(dk+dv)/time, masked pairs left out)", "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": f"{w.name} through fa_attention: B={B} H={H} Nq={Nq} Nk={Nk} dk={dk} dv={dv} "
                               f"{w.dtype}{' causal' if w.causal else ''}, {args.layout} storage",
                   "B": B, "H": H, "Nq": Nq, "Nk": Nk, "dk": dk, "dv": dv, "causal": w.causal,
                   "layout": args.layout, "parallelism": "replicas", "l2": l2_text},
        "roofline": roof,
        "e2e": None,  # the host-buffer entry point takes the contiguous self-attention form only
        "gpu_launches": launches["n"],
        "per_step_ms": step_spread(per),
        "kernel": "key-range split + combine" if ws_bytes else "one launch",
        "workspace_bytes": ws_bytes,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def bench_backward(args, w, world, rank, local_rank):
    """fa_backward on the workload: one step = dQ, dK, dV from (Q, K, V, O, dO,
    LSE) by recomputation; FLOPs counted as the five products of 2 N^2 d each
    per head (2.5 times the forward's), halved under the causal mask."""
    import torch
    import tiled_online_softmax_attn_gb300 as fa
    from tiled_online_softmax_attn_gb300 import build as fa_build
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa_build.build()
    q_np, k_np, v_np = w.inputs()
    g_np = synth.tensor(3 * w.seed + 9, w.shape, w.dtype)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q, k, v, g = (torch.from_numpy(x).to(tdt).to(dev) for x in (q_np, k_np, v_np, g_np))
    o, lse = fa.fa_forward(q, k, v, scale=w.scale, causal=w.causal)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws_bytes = fa.backward_workspace_size(*w.shape, tdt)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    n_launch, path = fa.backward_plan(*w.shape, tdt, w.causal, ws_bytes)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fa_backward(q, k, v, o, g, lse, scale=w.scale, causal=w.causal, dq=dq, dk=dk, dv=dv,
                       workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    # Q, K, V, O, dO and LSE are read
    in_bytes = 5 * q.numel() * q.element_size() + lse.numel() * lse.element_size()
    flush_bytes, l2_text = l2_plan(device_l2_bytes(torch, dev), in_bytes)
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device=dev) if flush_bytes else None
    if dist:
        dist.barrier()
    with ClockSampler(local_rank) as clocks:
        clocks.mark_start()
        ms_total, per = time_steps(torch, dev, stream, step, args.steps, flush)
        clocks.mark_end()
    if fa.check_device_error(stream.cuda_stream) != fa.FA_OK:
        raise RuntimeError(fa.last_error())
    ms = reduce_max(ms_total, dist, dev) / args.steps
    spread = step_spread(per)
    flops = 2.5 * w.flops
    value = world * flops / (ms * 1e-3) / 1e12
    peaks, peak_kind = load_peaks()
    peak = float(peaks["bf16_tflops"])
    line = {
        "metric": "attention bwd TFLOP/s (10·B·H·N²·d/time, halved for causal)", "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": workload_desc(w), "pass": "backward", "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "parallelism": "replicas", "l2": l2_text},
        "roofline": {"bound": "tensor", "achieved": value / world, "peak": peak, "unit": "TFLOP/s",
                     "frac": value / world / peak, "peak_source": peak_kind,
                     "note": "5 products counted; the kernels form S and dP twice (7 products)"},
        "gpu_launches": args.steps * n_launch,  # delta, (hi/lo split,) dK/dV, dQ
        "per_step_ms": spread,
        "kernel": path + " backward",
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="multihead", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--batch", type=int, help="override B of the workload (smaller profiling cases)")
    ap.add_argument("--heads", type=int, help="override H of the workload")
    ap.add_argument("--seq", type=int, help="override N (the query count) of the workload")
    ap.add_argument("--nk", type=int, help="key count for fa_attention (default: the query count)")
    ap.add_argument("--dv", type=int, help="value width for fa_attention (default: d)")
    ap.add_argument("--layout", choices=["bhnd", "bnhd"], help="time fa_attention on this storage "
                    "(bnhd: (batch, seq, heads, dim) seen through a transposed view)")
    ap.add_argument("--e2e-steps", type=int, default=20, help="0 skips the end-to-end measurement")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads of the timed oracle (0: all host cores)")
    ap.add_argument("--pass", dest="which", choices=["forward", "backward"], default="forward",
                    help="backward times fa_backward (dQ, dK, dV by recomputation from LSE)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = w.scaled(B=args.batch)
    if args.heads:
        w = w.scaled(H=args.heads)
    if args.seq:
        w = w.scaled(N=args.seq)

    if args.impl == "reference":
        if rank == 0:
            q, k, v = w.inputs()
            reference_arm(args, w, q, k, v, rank, world)
        return

    import torch
    import tiled_online_softmax_attn_gb300 as fa
    from tiled_online_softmax_attn_gb300 import build as fa_build

    if args.which == "backward":
        return bench_backward(args, w, world, rank, local_rank)
    if args.layout or args.nk or args.dv:
        args.layout = args.layout or "bhnd"
        return bench_attention(args, w, world, rank, local_rank)

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa_build.build()
    fa.load()

    q_np, k_np, v_np = w.inputs()
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q_h, k_h, v_h = (torch.from_numpy(x).to(tdt).pin_memory() for x in (q_np, k_np, v_np))
    q, k, v = (x.to(dev) for x in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty(w.shape[:3], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # the workspace lets wide heads (the fp32 d=1024 shape) use the tensor cores
    ws_bytes = fa.workspace_size(w.B, w.H, w.N, w.d, q.dtype, q.dtype, w.causal)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    per_call, path = fa.plan(w.B, w.H, w.N, w.d, q.dtype, q.dtype, w.causal, ws_bytes)
    launches = {"n": 0}

    def step():
        fa.fa_forward(q, k, v, o=o, lse=lse, scale=w.scale, causal=w.causal, stream=stream, workspace=ws)
        launches["n"] += per_call

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.check_device_error(stream.cuda_stream) != fa.FA_OK:
        raise RuntimeError(fa.last_error())

    flush_bytes, l2_text = l2_plan(device_l2_bytes(torch, dev), 3 * q.numel() * q.element_size())
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device=dev) if flush_bytes else None
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches["n"] = 0
    with ClockSampler(local_rank) as clocks:
        clocks.mark_start()
        ms_total, per = time_steps(torch, dev, stream, step, args.steps, flush)
        clocks.mark_end()
    if dist:
        dist.barrier()
    timed_launches = launches["n"]
    spread = step_spread(per)
    if fa.check_device_error(stream.cuda_stream) != fa.FA_OK:
        raise RuntimeError(fa.last_error())
    ms_total = reduce_max(ms_total, dist, dev)
    ms_step = ms_total / args.steps
    value = aggregate_tflops(w.flops, ms_step, world)

    # ---- end to end: host buffers through fa_forward_host, copies inside the timed region
    e2e = None
    if args.e2e_steps > 0:
        e2e = measure_e2e(args, w, fa, torch, dev, stream, q_h, k_h, v_h, q, o, lse, tdt, dist, world)
    line_e2e = e2e

    peaks, peak_kind = load_peaks()
    kernel_key = "tc" if path.startswith("tensor-core") else ("wide" if path.startswith("wide") else "general")
    # the roofline is the slower of the tensor-core time and the HBM time
    t_tensor = w.flops / (float(peaks["bf16_tflops"]) * 1e12)
    t_hbm = w.bytes / (float(peaks["hbm_gbs"]) * 1e9)
    if t_tensor >= t_hbm:
        peak = float(peaks["bf16_tflops"])
        achieved = w.flops / (ms_step * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak}
    else:
        peak = float(peaks["hbm_gbs"])
        achieved = w.bytes / (ms_step * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak}
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json, burst)" if peak_kind == "measured" else "fallback"
    roof["traffic"], roof["traffic_note"] = traffic_for(kernel_key, w)
    roof["algorithmic_bytes"] = w.bytes
    roof["algorithmic_flops"] = w.flops
    roof["launches_per_step"] = per_call
    if per_call > 1:
        roof["note"] = "achieved over the whole step (%d launches)" % per_call

    clock_summary = clocks.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": workload_desc(w), "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "seed": w.seed, "parallelism": "replicas",
                   "l2": l2_text},
        "pct_bf16_peak": 100.0 * (w.flops / (ms_step * 1e-3) / 1e12) / float(peaks["bf16_tflops"]),
        "pct_bf16_peak_sustained": 100.0 * (w.flops / (ms_step * 1e-3) / 1e12) / float(peaks["bf16_tflops_sustained"]),
        "roofline": roof,
        "exp_roofline": exp_roofline(w, ms_step, torch.cuda.get_device_properties(dev).multi_processor_count,
                                     clock_summary.get("sm_max_mhz")),
        "e2e": line_e2e,
        "gpu_launches": timed_launches,
        "per_step_ms": spread,
        "kernel": path,
        "workspace_bytes": ws_bytes,
        "clocks": clock_summary,
    }
    if rank == 0 and not args.no_cpu_baseline:
        rate, nrows, threads, el = oracle_rows_rate(w, q_np, k_np, v_np, args.cpu_seconds,
                                                    threads=args.cpu_threads)
        line["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"{nrows} seeded query rows of the workload (drawn with "
                                          f"replacement), full key range each, {el:.1f} s on "
                                          f"{threads} host threads"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
