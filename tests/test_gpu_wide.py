"""GPU parity of the wide-head tensor-core path (d = 128..1024, fp32 inputs as
bf16 hi + lo pairs, bf16 inputs with d >= 256), with and without a workspace
(split key ranges merged by the combine kernel, or one split)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_online_softmax_attn_gb300 as fa
from parity import compare

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}

WIDE = [
    (1, 1, 300, 128, "fp32", False),
    (1, 2, 333, 256, "fp32", True),
    (2, 1, 200, 384, "fp32", True),
    (1, 1, 640, 512, "fp32", False),
    (1, 2, 257, 512, "bf16", False),
    (1, 1, 500, 256, "bf16", True),
    (1, 1, 129, 1024, "bf16", True),
    (1, 1, 1, 1024, "fp32", False),
    # d = 512 and 1024 run as clusters sharing one formation of S
    (1, 3, 300, 512, "fp32", True),
    (2, 1, 1000, 1024, "fp32", False),
    (1, 2, 700, 1024, "fp32", True),
    (1, 1, 1000, 1024, "bf16", False),
    (2, 2, 77, 512, "bf16", True),
]


def run(w, ws_mode, o_dtype=None):
    q, k, v = w.inputs()
    tdt = TORCH_DT[w.dtype]
    odt = TORCH_DT[o_dtype or w.dtype]
    qd, kd, vd = (torch.from_numpy(x).cuda().to(tdt) for x in (q, k, v))
    need = fa.workspace_size(w.B, w.H, w.N, w.d, tdt, odt, w.causal)
    nbytes = {"full": need, "small": min(need, 1 << 20), "none": 0}[ws_mode]
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda") if nbytes else None
    launches, desc = fa.plan(w.B, w.H, w.N, w.d, tdt, odt, w.causal, nbytes)
    o, lse = fa.fa_forward(qd, kd, vd, scale=w.scale, causal=w.causal, o_dtype=odt, workspace=ws)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    o_ref, l_ref = oracle.attention(q, k, v, w.scale, w.causal)
    stats = compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, w.dtype, o_dtype or w.dtype)
    return desc, stats


@pytest.mark.parametrize("ws_mode", ["full", "small", "none"])
@pytest.mark.parametrize("B,H,N,d,dtype,causal", WIDE)
def test_wide_path(B, H, N, d, dtype, causal, ws_mode):
    w = synth.Workload("t", B, H, N, d, dtype, causal, seed=5000 + N + d)
    desc, _ = run(w, ws_mode)
    if dtype == "bf16" or ws_mode == "full":
        assert desc.startswith("wide-head"), desc
        assert ("cluster=%d" % (d // 256)) in desc if d in (512, 1024) else "cluster=1" in desc


def test_large_d_workload_on_tensor_cores():
    w = synth.WORKLOADS["large_d"]
    desc, stats = run(w, "full")
    assert "wide-head" in desc and "splits=" in desc
    assert stats["o_max"] <= 2e-4


def test_large_d_workload_bf16_output():
    desc, _ = run(synth.WORKLOADS["large_d"], "full", o_dtype="bf16")


def test_workspace_query_matches_plan():
    need = fa.workspace_size(1, 1, 1024, 1024, torch.float32, torch.float32)
    assert need > 0
    n, desc = fa.plan(1, 1, 1024, 1024, torch.float32, torch.float32, False, need)
    assert n == 3 and "hi+lo" in desc   # split pass, attention, combine
    # without a workspace fp32 inputs have nowhere to put their bf16 copies
    assert fa.plan(1, 1, 1024, 1024, torch.float32, torch.float32, False, 0)[1] == "general-d"
    assert fa.workspace_size(4, 32, 4096, 128, torch.bfloat16, torch.bfloat16) == 0


def test_host_buffer_path_with_wide_heads():
    w = synth.Workload("t", 2, 3, 300, 256, "fp32", True, seed=5100)
    q, k, v = w.inputs()
    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (q, k, v))
    oh = torch.empty(w.shape, dtype=torch.float32).pin_memory()
    lh = torch.empty(w.shape[:3], dtype=torch.float32).pin_memory()
    ws = torch.empty(fa.host_workspace_size(*w.shape, torch.float32, torch.float32), dtype=torch.uint8, device="cuda")
    fa.forward_host(qh, kh, vh, oh, lh, ws, scale=w.scale, causal=True)
    o_ref, l_ref = oracle.attention(q, k, v, w.scale, True)
    compare(oh.numpy(), lh.numpy(), o_ref, l_ref, "fp32", "fp32")
