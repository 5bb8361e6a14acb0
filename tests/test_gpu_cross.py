"""GPU parity of fa_attention: cross-attention shapes (Nq != Nk, dv != dk) and
strided layouts, against the CPU oracle.  The oracle always sees contiguous
copies; the kernels see the strided views."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_online_softmax_attn_gb300 as fa
from parity import compare

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


def draw(seed, B, H, Nq, Nk, dk, dv, dtype):
    q = synth.tensor(3 * seed, (B, H, Nq, dk), dtype)
    k = synth.tensor(3 * seed + 1, (B, H, Nk, dk), dtype)
    v = synth.tensor(3 * seed + 2, (B, H, Nk, dv), dtype)
    return q, k, v


def as_layout(x, layout, dtype):
    """A CUDA view with shape [B, H, N, d] of the array x in the given memory layout."""
    t = torch.from_numpy(np.ascontiguousarray(x)).to(TORCH_DT[dtype])
    if layout == "bhnd":
        return t.cuda()
    if layout == "bnhd":            # (batch, seq, heads, dim) storage
        return t.transpose(1, 2).contiguous().cuda().transpose(1, 2)
    if layout == "padded":          # rows padded to a wider buffer, heads interleaved
        B, H, N, d = t.shape
        buf = torch.zeros((B, N, H, d + 64), dtype=t.dtype)
        buf[..., :d] = t.transpose(1, 2)
        return buf.cuda().transpose(1, 2)[..., :d]
    raise ValueError(layout)


def check(seed, B, H, Nq, Nk, dk, dv, dtype, causal, layouts=("bhnd",) * 4, o_dtype=None):
    q, k, v = draw(seed, B, H, Nq, Nk, dk, dv, dtype)
    qd, kd, vd = (as_layout(x, lay, dtype) for x, lay in zip((q, k, v), layouts[:3]))
    odt = TORCH_DT[o_dtype or dtype]
    o = as_layout(np.zeros((B, H, Nq, dv), np.float32), layouts[3], o_dtype or dtype).to(odt)
    scale = 1.0 / np.sqrt(dk)
    fa.fa_attention(qd, kd, vd, o=o, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    lse = fa.fa_attention(qd, kd, vd, scale=scale, causal=causal)[1]
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, dtype, o_dtype or dtype)


CROSS = [
    # (B, H, Nq, Nk, dk, dv, dtype): tensor-core kernel dims and others
    (1, 2, 300, 700, 128, 128, "bf16"),
    (2, 1, 700, 300, 64, 64, "bf16"),
    (1, 2, 257, 129, 64, 128, "bf16"),
    (1, 2, 129, 257, 128, 64, "bf16"),
    (1, 1, 1, 500, 128, 128, "bf16"),
    (1, 1, 500, 1, 64, 64, "bf16"),
    (1, 2, 100, 333, 40, 72, "bf16"),     # padded to 64 / 128 on the tensor cores
    (2, 2, 190, 260, 96, 40, "bf16"),
    (1, 1, 77, 300, 120, 8, "bf16"),
    (2, 1, 150, 90, 96, 200, "fp32"),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk,dk,dv,dtype", CROSS)
def test_cross_attention_shapes(B, H, Nq, Nk, dk, dv, dtype, causal):
    check(7000 + Nq + Nk, B, H, Nq, Nk, dk, dv, dtype, causal)


LAYOUTS = [
    ("bnhd", "bnhd", "bnhd", "bnhd"),
    ("bnhd", "bhnd", "padded", "bhnd"),
    ("padded", "padded", "padded", "bnhd"),
]


@pytest.mark.parametrize("layouts", LAYOUTS)
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (64, 128), (80, 48)])
@pytest.mark.parametrize("causal", [False, True])
def test_strided_layouts(layouts, dk, dv, causal):
    check(7100 + dk + dv, 2, 3, 320, 280, dk, dv, "bf16", causal, layouts)


def test_strided_fp32_output():
    check(7200, 1, 4, 200, 200, 128, 128, "bf16", True, ("bnhd",) * 4, o_dtype="fp32")


def test_sequence_major_matches_contiguous_bitwise():
    """The tensor-core kernel gives the same bits whichever layout the tensors
    live in: only the addresses change."""
    q, k, v = draw(7300, 2, 4, 384, 384, 128, 128, "bf16")
    a = [as_layout(x, "bhnd", "bf16") for x in (q, k, v)]
    b = [as_layout(x, "bnhd", "bf16") for x in (q, k, v)]
    o1, l1 = fa.fa_attention(*a, causal=True)
    o2, l2 = fa.fa_attention(*b, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3, l3 = fa.fa_forward(*a, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
