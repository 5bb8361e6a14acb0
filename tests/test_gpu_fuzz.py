"""Seeded random sweep of the GPU paths against the oracle.

Each case draws a shape and options from a fixed seed (so every run checks the
same cases): batch, heads, ragged query and key lengths (cross-attention when
they differ), head dimensions (the tensor-core pairs and others), the causal
mask, the output dtype, scaled-up scores, the memory layout, and whether a
workspace is passed (which lets few-block problems take the key-range split).
The forward is compared with the fp64 oracle under the same tolerances as the
fixed cases; the backward with the gradient oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_online_softmax_attn_gb300 as fa
from parity import compare, half_ulp_bf16

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


def _layout(x, layout, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x)).to(TORCH_DT[dtype])
    if layout == "bhnd":
        return t.cuda()
    # (batch, seq, heads, dim) storage seen through a transposed view
    return t.transpose(1, 2).contiguous().cuda().transpose(1, 2)


def forward_case(i):
    rng = np.random.default_rng(91000 + i)
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    dk = int(rng.choice([64, 128, 64, 128, 32, 96]))
    dv = dk if rng.random() < 0.6 else int(rng.choice([64, 128]))
    Nq = int(rng.choice([1, 2, 127, 128, 129, 255, 256, 257]) if rng.random() < 0.4 else rng.integers(1, 700))
    cross = rng.random() < 0.5
    Nk = int(rng.integers(1, 900)) if cross else Nq
    causal = bool(rng.random() < 0.4)
    o_dtype = "fp32" if rng.random() < 0.25 else "bf16"
    mult = 4.0 if rng.random() < 0.25 else 1.0
    layout = "bnhd" if rng.random() < 0.3 else "bhnd"
    use_ws = bool(rng.random() < 0.5)
    return B, H, Nq, Nk, dk, dv, causal, o_dtype, mult, layout, use_ws


@pytest.mark.parametrize("i", range(32))
def test_random_forward(i):
    B, H, Nq, Nk, dk, dv, causal, o_dtype, mult, layout, use_ws = forward_case(i)
    seed = 92000 + i
    q = synth.tensor(3 * seed, (B, H, Nq, dk), "bf16") * mult
    k = synth.tensor(3 * seed + 1, (B, H, Nk, dk), "bf16") * mult
    v = synth.tensor(3 * seed + 2, (B, H, Nk, dv), "bf16")
    qd, kd, vd = (_layout(x, layout, "bf16") for x in (q, k, v))
    odt = TORCH_DT[o_dtype]
    scale = 1.0 / np.sqrt(dk)
    ws = None
    if use_ws:
        need = fa.attention_workspace_size(qd, kd, vd, causal=causal, o_dtype=odt)
        if need:
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o, lse = fa.fa_attention(qd, kd, vd, scale=scale, causal=causal, o_dtype=odt, workspace=ws)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", o_dtype)


def backward_case(i):
    rng = np.random.default_rng(93000 + i)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    d = int(rng.choice([64, 128, 64, 128, 32]))
    N = int(rng.choice([1, 127, 128, 129, 256]) if rng.random() < 0.4 else rng.integers(1, 600))
    causal = bool(rng.random() < 0.5)
    return B, H, N, d, causal


@pytest.mark.parametrize("i", range(12))
def test_random_backward(i):
    B, H, N, d, causal = backward_case(i)
    w = synth.Workload("fuzz", B, H, N, d, "bf16", causal, seed=94000 + i)
    q, k, v = w.inputs()
    dout = synth.tensor(3 * w.seed + 9, w.shape, "bf16")
    qd, kd, vd, gd = (torch.from_numpy(x).cuda().to(torch.bfloat16) for x in (q, k, v, dout))
    o, lse = fa.fa_forward(qd, kd, vd, scale=w.scale, causal=causal)
    grads = fa.fa_backward(qd, kd, vd, o, gd, lse, scale=w.scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    ref = oracle.attention_backward(q, k, v, dout, w.scale, causal)
    # dS = P (dP - delta) is a difference of two dot products of length d that
    # the GPU forms in different fp32 orders (the tensor core for dP, the delta
    # kernel for dO . O), so where the exact gradient vanishes (a single key:
    # P = 1, dP = delta) the result is their rounding difference: a floor of a
    # few fp32 ulps of d |dO| |v| |k| scale, far below 2e-2 of any gradient that
    # does not vanish
    floor = 4 * 2.0 ** -24 * d * np.abs(dout).max() * np.abs(v).max() * np.abs(k).max() * w.scale
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        g = g.float().cpu().numpy().astype(np.float64)
        bound = 2e-2 * np.abs(r).max() + half_ulp_bf16(r) + floor
        err = np.abs(g - r)
        assert np.all(err <= bound), f"{name}: max err {err.max():.3e} vs scale {np.abs(r).max():.3e}"
