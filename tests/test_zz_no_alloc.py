"""fa_forward_noalloc: the wide-head path for callers that cannot allocate
device memory while they run (a plugin whose host framework owns all GPU
memory, a service that fixes its memory plan before serving), with its
scratch in a fixed array inside the library.

Runs last (file name) so that a failure here cannot hide another test's.
Each case calls the allocation-free entry point through the C ABI and checks
its output against fa_forward_ws, the entry point that takes a caller
workspace, and against the CPU oracle, within the parity tolerances of the
other GPU tests, for two calls in a row: the second call reuses the array
the first one left behind.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_online_softmax_attn_gb300 as fa
from parity import compare

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}
CODE = {"bf16": fa.FA_BF16, "fp32": fa.FA_FP32}


def noalloc(q, k, v, o, lse, w):
    lib = fa.load()
    return lib.fa_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  w.B, w.H, w.N, w.d, w.scale, int(w.causal), CODE[w.dtype], CODE[w.dtype],
                                  torch.cuda.current_stream().cuda_stream)


def with_workspace(q, k, v, w):
    tdt = TORCH_DT[w.dtype]
    ws = torch.empty(fa.workspace_size(w.B, w.H, w.N, w.d, tdt, tdt, w.causal), dtype=torch.uint8, device="cuda")
    return fa.fa_forward(q, k, v, scale=w.scale, causal=w.causal, workspace=ws)


def one_call(w):
    q_np, k_np, v_np = w.inputs()
    q, k, v = (torch.from_numpy(x).cuda().to(TORCH_DT[w.dtype]) for x in (q_np, k_np, v_np))
    o = torch.empty_like(q)
    lse = torch.empty(w.shape[:3], dtype=torch.float32, device="cuda")
    st = noalloc(q, k, v, o, lse, w)
    assert st == fa.FA_OK, fa.last_error()
    o_ws, lse_ws = with_workspace(q, k, v, w)
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    got_o, got_l = o.float().cpu().numpy(), lse.cpu().numpy()
    compare(got_o, got_l, o_ws.float().cpu().numpy().astype(np.float64),
            lse_ws.cpu().numpy().astype(np.float64), w.dtype, w.dtype)
    o_ref, lse_ref = oracle.attention(q_np, k_np, v_np, w.scale, w.causal)
    compare(got_o, got_l, o_ref, lse_ref, w.dtype, w.dtype)


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    # the fp32 d = 1024 shape (about 29 MB of scratch) and then a causal bf16
    # d = 256 shape with new data, on the scratch the first call left behind
    one_call(synth.WORKLOADS["large_d"])
    one_call(synth.Workload("t", 2, 3, 700, 256, "bf16", True, seed=6001))


def test_the_same_problem_twice():
    w = synth.Workload("t", 1, 2, 513, 512, "fp32", False, seed=6002)
    one_call(w)
    one_call(w.scaled(seed=6003))


def test_problem_that_fits_only_without_key_splits():
    """fp32, d = 1024, N = 2048: the bf16 hi/lo copies take 24 MB, and the
    partials of a key split would push the scratch past its 32 MB, so the
    call plans a single key range; fa_forward_ws with a full workspace splits
    the keys, so the two agree to rounding, and both match the oracle."""
    w = synth.Workload("t", 1, 1, 2048, 1024, "fp32", False, seed=6004)
    full = fa.workspace_size(w.B, w.H, w.N, w.d, fa.FA_FP32, fa.FA_FP32, False)
    assert full > (32 << 20)
    assert "splits=1" in fa.plan(w.B, w.H, w.N, w.d, fa.FA_FP32, fa.FA_FP32, False, 32 << 20)[1]
    one_call(w)
    one_call(w.scaled(seed=6005))


def test_problems_beyond_the_scratch_are_rejected():
    # fp32, d = 1024, 8 heads of 4096: ~400 MB of bf16 copies alone
    w = synth.Workload("t", 1, 8, 4096, 1024, "fp32", False, seed=1)
    # placeholder addresses, far apart and never dereferenced: the size check
    # rejects the call before anything is launched
    q, k, v, o = (i << 44 for i in (1, 2, 3, 4))
    lib = fa.load()
    st = lib.fa_forward_noalloc(q, k, v, o, None, w.B, w.H, w.N, w.d, w.scale, 0, fa.FA_FP32, fa.FA_FP32, None)
    assert st == fa.FA_ERR_UNSUPPORTED
    assert "maximum" in fa.last_error()


def test_other_paths_are_not_covered():
    q = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lib = fa.load()
    st = lib.fa_forward_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), None,
                                1, 1, 64, 128, 0.1, 0, fa.FA_BF16, fa.FA_BF16, None)
    assert st == fa.FA_ERR_UNSUPPORTED and "wide-head" in fa.last_error()
