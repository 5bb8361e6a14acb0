"""GPU parity of the backward pass against the fp64 gradient oracle.

Tolerance (the pages fix none): the GPU recomputes the weights from the
forward's LSE and forms delta_i = dO_i . O_i from the forward's stored O.
With bf16 inputs O is stored in bf16 (relative rounding 2^-9) and every
product runs on bf16 operands with fp32 accumulation, so each gradient
element carries an error of a few 2^-9 of the gradient's scale: the bound is
max|g_gpu - g_ref| <= 2e-2 * max|g_ref| (about 10 half-ulps of bf16) plus,
for bf16 gradient storage, half a bf16 ulp of the element.  fp32 inputs keep
fp32 throughout: 1e-5 * max|g_ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_online_softmax_attn_gb300 as fa
from parity import half_ulp_bf16, sample_rows

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}
REL = {"bf16": 2e-2, "fp32": 1e-5}
# fp32 inputs on the tensor cores travel as bf16 hi + lo pairs (16 significant
# bits of each operand, the lo*lo term dropped: about 2^-16 of each product),
# for the weights and dS as well: ten such units of the gradient's scale.
REL_FP32_TC = 1.5e-4


def _rel(dtype, path):
    return REL_FP32_TC if dtype == "fp32" and "tensor-core" in path else REL[dtype]


def _check(grads, ref, dtype, grad_dtype, path="general"):
    stats = {}
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        if np.size(r) == 0:
            continue
        g = np.asarray(g, dtype=np.float64)
        err = np.abs(g - r)
        bound = _rel(dtype, path) * np.abs(r).max()
        if grad_dtype == "bf16":
            bound = bound + half_ulp_bf16(r)
        stats[name] = (float(err.max()), float(np.abs(r).max()))
        assert np.all(err <= bound), f"{name}: max err {err.max():.3e} vs scale {np.abs(r).max():.3e}"
    return stats


def _gpu_backward(w, q, k, v, dout, grad_dtype=None):
    tdt = TORCH_DT[w.dtype]
    qd, kd, vd, gd = (torch.from_numpy(x).cuda().to(tdt) for x in (q, k, v, dout))
    o, lse = fa.fa_forward(qd, kd, vd, scale=w.scale, causal=w.causal)
    gdt = TORCH_DT[grad_dtype or w.dtype]
    dq, dk, dv = fa.fa_backward(qd, kd, vd, o, gd, lse, scale=w.scale, causal=w.causal, grad_dtype=gdt)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    return dq, dk, dv


def run_backward(B, H, N, d, dtype, causal, grad_dtype=None, seed=0):
    w = synth.Workload("t", B, H, N, d, dtype, causal, seed=seed)
    q, k, v = w.inputs()
    dout = synth.tensor(3 * seed + 9, w.shape, dtype)
    path = fa.backward_plan(B, H, N, d, TORCH_DT[dtype], causal)[1]
    grads = _gpu_backward(w, q, k, v, dout, grad_dtype)
    ref = oracle.attention_backward(q, k, v, dout, w.scale, causal)
    return _check([g.float().cpu().numpy() for g in grads], ref, dtype, grad_dtype or dtype, path), path


SHAPES = [
    (1, 2, 100, 64, "bf16"),
    (2, 1, 257, 128, "bf16"),
    (1, 1, 300, 40, "fp32"),
    (1, 2, 64, 16, "fp32"),
    (1, 1, 1, 64, "bf16"),
    (1, 2, 640, 128, "bf16"),
    (1, 2, 384, 64, "bf16"),
    (1, 1, 130, 256, "fp32"),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d,dtype", SHAPES)
def test_backward_matches_oracle(B, H, N, d, dtype, causal):
    run_backward(B, H, N, d, dtype, causal, seed=8000 + N + d)


WIDE = [
    # (B, H, N, d, dtype): heads too wide for one tile's gradients in tensor memory
    (1, 2, 300, 256, "bf16"),
    (1, 1, 200, 512, "bf16"),
    (1, 1, 129, 1024, "bf16"),
    (1, 2, 150, 128, "fp32"),
    (1, 1, 257, 256, "fp32"),
    (2, 1, 64, 384, "fp32"),
    (1, 1, 130, 1024, "fp32"),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d,dtype", WIDE)
def test_wide_head_backward_on_tensor_cores(B, H, N, d, dtype, causal):
    """The wide-head tensor-core backward (a CTA per gradient column slice,
    the score products over the whole head dimension) against the oracle."""
    stats, path = run_backward(B, H, N, d, dtype, causal, seed=8300 + N + d)
    assert path.startswith("wide-head tensor-core"), path
    if dtype == "fp32":
        print(f"wide fp32 d={d} causal={causal}: " +
              ", ".join(f"{k} {e / m:.2e}" for k, (e, m) in stats.items()))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(300, 8), (200, 40), (257, 80), (130, 96), (513, 120)])
def test_narrow_head_backward_on_tensor_cores(N, d, causal):
    """bf16 heads narrower than 64 or between 64 and 128 (multiples of 8):
    the tensor-core backward loads them padded with zero columns and writes
    only their own columns of dQ, dK and dV."""
    stats, path = run_backward(1, 2, N, d, "bf16", causal, seed=8400 + N + d)
    assert path == "tensor-core", path


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", [(2, 80, 300, 64), (2, 80, 300, 128), (1, 80, 2000, 128), (2, 40, 513, 40),
                                     (1, 8, 3000, 64)])
def test_persistent_backward_ctas(B, H, N, d, causal):
    """More items (128-row tiles x heads) than SMs, each of at most 2048
    tile-columns (16 tiles at d = 128, 32 at d = 64): the dK/dV and dQ kernels
    run on persistent CTAs that loop over items, handing the resident tiles and
    the accumulators over between them.  Every gradient element against the
    oracle."""
    n_t, width = (N + 127) // 128, 64 if d <= 64 else 128
    assert n_t * width <= 2048 and n_t * B * H > 152
    stats, path = run_backward(B, H, N, d, "bf16", causal, seed=8600 + N + d)
    assert path == "tensor-core", path


def test_persistent_backward_leaves_neighbouring_memory_alone():
    """dQ, dK and dV of 480 persistent items inside sentinel-filled buffers."""
    B, H, N, d = 2, 80, 300, 64
    w = synth.Workload("t", B, H, N, d, "bf16", False, seed=8650)
    q, k, v = w.inputs()
    dout = synth.tensor(3 * 8650 + 9, w.shape, "bf16")
    qt, kt, vt, gt = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (q, k, v, dout))
    o, lse = fa.fa_forward(qt, kt, vt, scale=w.scale)
    n, guard = B * H * N * d, 256
    bufs = [torch.full((n + 2 * guard,), 0x5A5A, dtype=torch.int16, device="cuda") for _ in range(3)]
    grads = [b[guard:guard + n].view(torch.bfloat16).view(w.shape) for b in bufs]
    fa.fa_backward(qt, kt, vt, o, gt, lse, scale=w.scale, dq=grads[0], dk=grads[1], dv=grads[2])
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    for b in bufs:
        h = b.cpu()
        assert bool((h[:guard] == 0x5A5A).all()) and bool((h[guard + n:] == 0x5A5A).all())
    ref = oracle.attention_backward(q, k, v, dout, w.scale, False)
    _check([g.float().cpu().numpy() for g in grads], ref, "bf16", "bf16", "tensor-core")


def test_narrow_head_backward_leaves_neighbouring_memory_alone():
    """dQ, dK and dV of a d = 40 head sit inside sentinel-filled buffers; the
    padded columns the kernel computes must not reach memory."""
    B, H, N, d = 1, 2, 300, 40
    w = synth.Workload("t", B, H, N, d, "bf16", True, seed=8450)
    q, k, v = w.inputs()
    dout = synth.tensor(3 * 8450 + 9, w.shape, "bf16")
    qt, kt, vt, gt = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (q, k, v, dout))
    o, lse = fa.fa_forward(qt, kt, vt, scale=w.scale, causal=True)
    n, guard = B * H * N * d, 256
    bufs = [torch.full((n + 2 * guard,), 0x5A5A, dtype=torch.int16, device="cuda") for _ in range(3)]
    grads = [b[guard:guard + n].view(torch.bfloat16).view(w.shape) for b in bufs]
    fa.fa_backward(qt, kt, vt, o, gt, lse, scale=w.scale, causal=True, dq=grads[0], dk=grads[1], dv=grads[2])
    torch.cuda.synchronize()
    for b in bufs:
        h = b.cpu()
        assert bool((h[:guard] == 0x5A5A).all()) and bool((h[guard + n:] == 0x5A5A).all())
    ref = oracle.attention_backward(q, k, v, dout, w.scale, True)
    _check([g.float().cpu().numpy() for g in grads], ref, "bf16", "bf16", "tensor-core")


def test_wide_fp32_backward_without_room_for_copies_runs_on_cuda_cores():
    B, H, N, d = 1, 1, 100, 256
    base = fa.load().fa_backward_workspace_size(B, H, N, d)
    assert fa.backward_workspace_size(B, H, N, d, torch.float32) > base
    assert fa.backward_plan(B, H, N, d, torch.float32, False, base)[1] == "general"
    assert fa.backward_plan(B, H, N, d, torch.bfloat16, False, base)[1].startswith("wide-head")


def test_backward_fp32_gradients_from_bf16_inputs():
    run_backward(1, 2, 200, 128, "bf16", True, grad_dtype="fp32", seed=8100)


def test_backward_is_deterministic():
    B, H, N, d = 1, 2, 300, 64
    x = [torch.randn(B, H, N, d, device="cuda", dtype=torch.bfloat16) for _ in range(4)]
    o, lse = fa.fa_forward(*x[:3], causal=True)
    a = fa.fa_backward(*x[:3], o, x[3], lse, causal=True)
    b = fa.fa_backward(*x[:3], o, x[3], lse, causal=True)
    torch.cuda.synchronize()
    for u, w in zip(a, b):
        assert torch.equal(u, w)


def test_full_size_multihead_backward_heads():
    """The multi-head workload at full size (B=4, H=32, N=4096, d=128, the
    inputs and launch the backward benchmark times): three whole heads, from
    different batches and head indices, against the gradient oracle (every
    dQ, dK and dV element of those heads)."""
    w = synth.WORKLOADS["multihead"]
    q, k, v = w.inputs()
    dout = synth.tensor(3 * w.seed + 9, w.shape, w.dtype)
    grads = _gpu_backward(w, q, k, v, dout)
    heads = [(0, 0), (1, 17), (3, 31)]

    def pick(x):
        return np.stack([x[b, h] for b, h in heads])[None]

    got = [pick(g.float().cpu().numpy()) for g in grads]
    ref = oracle.attention_backward(pick(q), pick(k), pick(v), pick(dout), w.scale, False)
    _check(got, ref, w.dtype, w.dtype)


@pytest.mark.parametrize("name,key_heads", [("causal", 2), ("peaked", 0)])
def test_full_size_backward_sampled(name, key_heads):
    """The causal (1x32x16384x128) and peaked (1x8x65536x64, Q and K x 4)
    workloads at full size, in the launch the backward benchmark times: dQ of
    sampled query rows in every head (rows 0, N-1, tile edges and a seeded
    draw) and, for the causal workload, dK and dV of sampled keys in the
    first and last head (a key's gradients sum over all queries of its head,
    so a head with a sampled key costs the oracle a full forward)."""
    w = synth.WORKLOADS[name]
    q, k, v = w.inputs()
    dout = synth.tensor(3 * w.seed + 9, w.shape, w.dtype)
    dq, dk, dv = (g.float().cpu().numpy().reshape(-1, w.d) for g in _gpu_backward(w, q, k, v, dout))
    rows = sample_rows(w.B, w.H, w.N, 192, seed=w.seed)
    rng = np.random.default_rng(w.seed + 1)
    keys = []
    for bh in [0, w.B * w.H - 1][:key_heads]:
        picks = [0, 1, 127, 128, w.N // 2, w.N - 129, w.N - 128, w.N - 1]
        keys += [bh * w.N + j for j in picks] + list(bh * w.N + rng.integers(0, w.N, size=12))
    keys = np.unique(np.array(keys, dtype=np.int64))
    ref = oracle.attention_backward_sampled(q, k, v, dout, w.scale, w.causal, rows, keys)
    _check([dq[rows], dk[keys], dv[keys]], ref, w.dtype, w.dtype)
