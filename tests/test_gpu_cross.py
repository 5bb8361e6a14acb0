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



SINGLE_TILE = [
    # (B, H, Nq, Nk, dk, dv, o_dtype): at most 128 query rows, so every item is
    # one query tile; Nk up to 64 key tiles runs persistent CTAs, beyond that one
    # CTA per item
    (1, 3, 1, 700, 128, 128, "bf16"),
    (2, 2, 100, 129, 64, 64, "bf16"),
    (1, 2, 128, 8192, 64, 128, "bf16"),
    (1, 2, 77, 9000, 128, 64, "bf16"),
    (3, 1, 128, 1, 64, 64, "fp32"),        # one key tile: no odd tiles to merge
    (1, 1, 33, 8321, 64, 64, "fp32"),
]


@pytest.mark.parametrize("B,H,Nq,Nk,dk,dv,o_dtype", SINGLE_TILE)
def test_single_query_tile_items(B, H, Nq, Nk, dk, dv, o_dtype):
    """Queries that fit one 128-row tile: the two softmax warpgroups take the
    even and the odd key tiles and their partial results are merged in the CTA.
    Checked against the oracle, with and without a workspace (key-range split
    where the plan picks one)."""
    q, k, v = draw(7500 + Nq + Nk, B, H, Nq, Nk, dk, dv, "bf16")
    qd, kd, vd = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (q, k, v))
    odt = TORCH_DT[o_dtype]
    scale = 1.0 / np.sqrt(dk)
    o, lse = fa.fa_attention(qd, kd, vd, scale=scale, o_dtype=odt)
    ws = torch.empty(max(1, fa.attention_workspace_size(qd, kd, vd, o_dtype=odt)), dtype=torch.uint8, device="cuda")
    o2, lse2 = fa.fa_attention(qd, kd, vd, scale=scale, o_dtype=odt, workspace=ws)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    o_ref, l_ref = oracle.attention(q, k, v, scale, False)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", o_dtype)
    compare(o2.float().cpu().numpy(), lse2.cpu().numpy(), o_ref, l_ref, "bf16", o_dtype)


@pytest.mark.parametrize("Nq,Nk,dk,dv", [(1, 800, 128, 128), (77, 800, 64, 64), (128, 640, 64, 128)])
def test_single_query_tile_key_range_split(Nq, Nk, dk, dv):
    """Key-range splits of single-tile items, uneven ones included: 800 keys
    are 7 key tiles, split 3 + 3 + 1 (the last range has no odd tile); 640 keys
    are 5, split 3 + 2."""
    q, k, v = draw(7600 + Nq + dk, 1, 1, Nq, Nk, dk, dv, "bf16")
    qd, kd, vd = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (q, k, v))
    ws_bytes = fa.attention_workspace_size(qd, kd, vd)
    assert ws_bytes > 0, "the problem should plan a key-range split"
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    scale = 1.0 / np.sqrt(dk)
    o, lse = fa.fa_attention(qd, kd, vd, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    o_ref, l_ref = oracle.attention(q, k, v, scale, False)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", "bf16")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hot", [3, 200, 300, 1000])
def test_single_query_tile_hot_key(d, hot):
    """One key whose score is about 40 above every other: in an even key tile
    (keys 3 and 300: tiles 0 and 2), an odd one (key 200: tile 1) or the ragged
    last one (key 1000 of 1001: tile 7).  The merge then weighs one warpgroup's partial result by about
    2^-58 against the other's, and O must be that key's V row."""
    B, H, Nq, Nk = 1, 2, 9, 1001
    q, k, v = draw(7700 + hot + d, B, H, Nq, Nk, d, d, "bf16")
    k = (k * 0.25).astype(np.float32)          # ordinary scores about 0.25 sigma
    u = np.zeros(d, np.float32)
    u[:8] = 4.0
    q[..., :8] = 4.0                            # every query row shares the direction u
    k[:, :, hot, :] = 0.0
    k[:, :, hot, :8] = u[:8] * (np.sqrt(d) * 40.0 / (8 * 16.0 * 4.0) * 4.0)
    q, k, v = (torch.from_numpy(x).to(torch.bfloat16).float().numpy() for x in (q, k, v))
    qd, kd, vd = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (q, k, v))
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_attention(qd, kd, vd, scale=scale)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    o_ref, l_ref = oracle.attention(q, k, v, scale, False)
    s_hot = scale * (q[0, 0, 0] @ k[0, 0, hot])
    assert s_hot > 30.0                         # the hot key dominates the row
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", "bf16")
    assert np.abs(o_ref[:, :, :, :] - v[:, :, hot:hot + 1, :]).max() < 1e-6


@pytest.mark.parametrize("B,H,Nq,Nk,dk,dv", [
    (4, 64, 64, 1000, 64, 64),      # 256 items, 8 key tiles: CTAs with two items (d_v = 64)
    (4, 64, 100, 700, 128, 128),    # the same at d_v = 128
    (2, 96, 128, 300, 128, 64),     # 192 items, 3 key tiles: odd count per warpgroup pair
    (8, 32, 77, 100, 64, 128),      # 256 items of one key tile: no odd tiles to merge
])
def test_single_query_tile_items_on_persistent_ctas(B, H, Nq, Nk, dk, dv):
    """More single-tile items than SMs: persistent CTAs take two items each, so
    the hand-over barriers (query tile, O columns, the merge's m/l/dq slots)
    change phase between items.  Every head checked against the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * H > sms and -(-Nk // 128) <= 64
    q, k, v = draw(7800 + Nq + Nk + dk, B, H, Nq, Nk, dk, dv, "bf16")
    qd, kd, vd = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (q, k, v))
    scale = 1.0 / np.sqrt(dk)
    o, lse = fa.fa_attention(qd, kd, vd, scale=scale)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    o_ref, l_ref = oracle.attention(q, k, v, scale, False)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", "bf16")
