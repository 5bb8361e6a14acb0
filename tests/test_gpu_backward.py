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
from parity import half_ulp_bf16

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}
REL = {"bf16": 2e-2, "fp32": 1e-5}


def run_backward(B, H, N, d, dtype, causal, grad_dtype=None, seed=0):
    w = synth.Workload("t", B, H, N, d, dtype, causal, seed=seed)
    q, k, v = w.inputs()
    dout = synth.tensor(3 * seed + 9, w.shape, dtype)
    tdt = TORCH_DT[dtype]
    qd, kd, vd, gd = (torch.from_numpy(x).cuda().to(tdt) for x in (q, k, v, dout))
    o, lse = fa.fa_forward(qd, kd, vd, scale=w.scale, causal=causal)
    gdt = TORCH_DT[grad_dtype or dtype]
    dq, dk, dv = fa.fa_backward(qd, kd, vd, o, gd, lse, scale=w.scale, causal=causal, grad_dtype=gdt)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    ref = oracle.attention_backward(q, k, v, dout, w.scale, causal)
    stats = {}
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = g.float().cpu().numpy().astype(np.float64)
        err = np.abs(g - r)
        bound = REL[dtype] * np.abs(r).max()
        if (grad_dtype or dtype) == "bf16":
            bound = bound + half_ulp_bf16(r)
        stats[name] = (float(err.max()), float(np.abs(r).max()))
        assert np.all(err <= bound), f"{name}: max err {err.max():.3e} vs scale {np.abs(r).max():.3e}"
    return stats


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
