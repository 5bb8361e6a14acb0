"""GPU parity of the key-range split of the tensor-core kernel: problems with
too few 256-row query blocks to fill the GPU (decode-like cross-attention,
short-query long-key self-attention) run with a workspace as CTAs over
(query block, key range) pairs whose partial O, maximum and sums a combine
step merges ("FlashAttention Engine: Hardware-Aware Exact Attention & SRAM
Tiling", "Core FlashAttention Mechanics", item 3).  Checked against the CPU
oracle, and against the same call without a workspace (no split)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_online_softmax_attn_gb300 as fa
from parity import compare

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


def draw(seed, B, H, Nq, Nk, dk, dv):
    q = synth.tensor(3 * seed, (B, H, Nq, dk), "bf16")
    k = synth.tensor(3 * seed + 1, (B, H, Nk, dk), "bf16")
    v = synth.tensor(3 * seed + 2, (B, H, Nk, dv), "bf16")
    return q, k, v


SPLIT = [
    # (B, H, Nq, Nk, dk, dv, o_dtype): one or two query blocks per head, long key ranges
    (1, 4, 256, 8192, 128, 128, "bf16"),
    (1, 2, 200, 8000, 64, 64, "bf16"),      # ragged queries and keys
    (2, 1, 512, 6000, 128, 64, "fp32"),     # fp32 O through the combine
    (1, 3, 1, 4096, 64, 128, "bf16"),       # a single query row per head
]


@pytest.mark.parametrize("B,H,Nq,Nk,dk,dv,o_dtype", SPLIT)
def test_split_matches_oracle_and_unsplit_call(B, H, Nq, Nk, dk, dv, o_dtype):
    q, k, v = draw(7300 + Nk % 97, B, H, Nq, Nk, dk, dv)
    qd, kd, vd = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (q, k, v))
    scale = 1.0 / np.sqrt(dk)
    odt = TORCH_DT[o_dtype]
    ws_bytes = fa.attention_workspace_size(qd, kd, vd, o_dtype=odt)
    assert ws_bytes > 0, "the problem should plan a key-range split"
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    o, lse = fa.fa_attention(qd, kd, vd, scale=scale, o_dtype=odt, workspace=ws)
    o1, lse1 = fa.fa_attention(qd, kd, vd, scale=scale, o_dtype=odt)  # no workspace: one CTA per block
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    o_ref, l_ref = oracle.attention(q, k, v, scale, False)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", o_dtype)
    compare(o1.float().cpu().numpy(), lse1.cpu().numpy(), o_ref, l_ref, "bf16", o_dtype)


def test_self_attention_workspace_entry_point_splits():
    """fa_forward_ws on [B, H, N, d] with the workspace fa_workspace_size asks
    for: fa_plan reports the split, and the result matches the oracle."""
    w = synth.Workload("split", 1, 2, 1024, 128, "bf16", False, seed=7400)
    need = fa.workspace_size(w.B, w.H, w.N, w.d, torch.bfloat16, torch.bfloat16, False)
    assert need > 0
    launches, desc = fa.plan(w.B, w.H, w.N, w.d, torch.bfloat16, torch.bfloat16, False, need)
    assert launches == 2 and "key splits" in desc, desc
    assert fa.plan(w.B, w.H, w.N, w.d, torch.bfloat16, torch.bfloat16, False, 0)[0] == 1
    q, k, v = w.inputs()
    qd, kd, vd = (torch.from_numpy(x).to(torch.bfloat16).cuda() for x in (q, k, v))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o, lse = fa.fa_forward(qd, kd, vd, scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    o_ref, l_ref = oracle.attention(q, k, v, w.scale, False)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16", "bf16")


def test_causal_and_full_gpu_problems_do_not_split():
    big = fa.workspace_size(4, 32, 4096, 128, torch.bfloat16, torch.bfloat16, False)
    causal = fa.workspace_size(1, 2, 8192, 128, torch.bfloat16, torch.bfloat16, True)
    assert big == 0 and causal == 0
