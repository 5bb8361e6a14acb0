"""Guard bands around the outputs: nothing outside O and LSE changes.

The result is exact up to rounding ("FlashAttention", ai360xpert.com, "Show
Me the Code"), and it goes to O and LSE only.  Each case places O and LSE
inside larger buffers: a band of sentinel elements before and after each,
and, for a strided O, sentinel rows after every head's rows and sentinel
columns after every row.  O and LSE themselves start as NaN, so an element
the call leaves unwritten fails the oracle comparison.  After the call every
sentinel element must hold its old bits, and O and LSE must match the
oracle.  Ragged N (1, 77, 129, 300, 513, 1000) puts the last query and key
tiles past the end of each head, where the kernels mask their stores.

Paths: the 64/128 tensor-core kernel (one work item per CTA, persistent
CTAs over many items, unmasked and causal, the key-range split with a
workspace), the general-d
kernel, the wide-head path (bf16 d = 256, fp32 d = 128 with key splits, and the
cluster form for d = 512 and 1024),
fa_attention with a padded O, fa_forward_host on host buffers and
fa_forward_noalloc.
"""
import math

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
BITS = {torch.bfloat16: torch.int16, torch.float32: torch.int32}
SENTINEL = {torch.int16: 0x5A5A, torch.int32: 0x5A5A5A5A}   # finite in both types
NAN_BITS = {torch.int16: 0x7FC0, torch.int32: 0x7FC00000}
GUARD = 640          # elements of sentinel before and after (1.25 / 2.5 KB)
RAGGED = [1, 77, 129, 300, 513, 1000]


class Guarded:
    """A tensor of `shape` and `dtype` inside a buffer of sentinel bits.

    `pad` = (rows, columns) adds sentinel rows after every head's rows and
    sentinel columns after every row (4-D shapes); the view is then strided.
    `where` is "cuda" or "pinned" (page-locked host memory)."""

    def __init__(self, shape, dtype, pad=(0, 0), where="cuda"):
        ib = BITS[dtype]
        self.ib = ib
        inner = list(shape)
        if len(shape) == 4:
            inner[2] += pad[0]
            inner[3] += pad[1]
        n = math.prod(inner)
        flat = torch.full((2 * GUARD + n,), SENTINEL[ib], dtype=ib)
        self.flat = flat.cuda() if where == "cuda" else flat.pin_memory()
        body = self.flat[GUARD:GUARD + n].view(inner)
        self.bits = body[:, :, :shape[2], :shape[3]] if len(shape) == 4 else body
        self.bits.fill_(NAN_BITS[ib])
        self.t = self.bits.view(dtype)

    def assert_intact(self, what):
        host = self.flat.cpu().clone()
        outside = torch.ones(host.numel(), dtype=torch.bool)
        off = self.bits.storage_offset() - self.flat.storage_offset()
        torch.as_strided(outside, self.bits.size(), self.bits.stride(), off).fill_(False)
        changed = (host[outside] != SENTINEL[self.ib]).nonzero().flatten()
        assert changed.numel() == 0, \
            f"{what}: {changed.numel()} sentinel elements changed, first at buffer index {int(changed[0])}"


def inputs(w, where="cuda"):
    q, k, v = w.inputs()
    tdt = TORCH_DT[w.dtype]
    ts = [torch.from_numpy(x).to(tdt) for x in (q, k, v)]
    ts = [t.cuda() for t in ts] if where == "cuda" else [t.pin_memory() for t in ts]
    return (q, k, v), ts


def finish(w, o, lse, host_inputs, o_dtype):
    torch.cuda.synchronize()
    assert fa.check_device_error() == fa.FA_OK, fa.last_error()
    o.assert_intact("O")
    lse.assert_intact("LSE")
    o_ref, lse_ref = oracle.attention(*host_inputs, w.scale, w.causal)
    compare(o.t.float().cpu().numpy(), lse.t.cpu().numpy(), o_ref, lse_ref, w.dtype, o_dtype)


def device_case(w, flags=0, workspace=False, o_dtype=None, expect_plan=None):
    o_dtype = o_dtype or w.dtype
    host_in, (q, k, v) = inputs(w)
    o = Guarded(w.shape, TORCH_DT[o_dtype])
    lse = Guarded(w.shape[:3], torch.float32)
    ws = None
    if workspace:
        nbytes = fa.workspace_size(w.B, w.H, w.N, w.d, CODE[w.dtype], CODE[o_dtype], w.causal)
        assert nbytes > 0
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        if expect_plan:
            assert expect_plan in fa.plan(w.B, w.H, w.N, w.d, CODE[w.dtype], CODE[o_dtype], w.causal, nbytes)[1]
    fa.fa_forward(q, k, v, o=o.t, lse=lse.t, scale=w.scale, causal=w.causal, flags=flags, workspace=ws)
    finish(w, o, lse, host_in, o_dtype)


@pytest.mark.parametrize("N", RAGGED)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_tensor_core_kernel(N, d, causal):
    device_case(synth.Workload("guard", 1, 2, N, d, "bf16", causal, seed=8000 + N + d))


@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_kernel_persistent_ctas(d):
    # 2 x 80 heads of three 256-row blocks: 480 items, several per CTA
    device_case(synth.Workload("guard", 2, 80, 513, d, "bf16", False, seed=8100 + d))


@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_kernel_persistent_causal_ctas(d):
    # 2 x 80 causal heads of two 256-row blocks (the second ragged): 320 short
    # items of unequal length on persistent CTAs
    device_case(synth.Workload("guard", 2, 80, 300, d, "bf16", True, seed=8150 + d))


@pytest.mark.parametrize("N", [513, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_key_range_split(N, d):
    device_case(synth.Workload("guard", 1, 1, N, d, "bf16", False, seed=8200 + N + d), workspace=True,
                expect_plan="key splits")


@pytest.mark.parametrize("N", RAGGED)
@pytest.mark.parametrize("causal", [False, True])
def test_general_kernel(N, causal):
    device_case(synth.Workload("guard", 1, 2, N, 40, "bf16", causal, seed=8300 + N),
                flags=fa.FA_FLAG_GENERAL_PATH)


@pytest.mark.parametrize("N", [1, 129, 513])
@pytest.mark.parametrize("causal", [False, True])
def test_wide_head_bf16(N, causal):
    device_case(synth.Workload("guard", 1, 2, N, 256, "bf16", causal, seed=8400 + N))


@pytest.mark.parametrize("N", [77, 300, 1000])
def test_wide_head_fp32_with_key_splits(N):
    device_case(synth.Workload("guard", 1, 1, N, 128, "fp32", False, seed=8500 + N), workspace=True,
                o_dtype="fp32", expect_plan="wide-head")


@pytest.mark.parametrize("N", [129, 1000])
@pytest.mark.parametrize("d,dtype", [(512, "fp32"), (1024, "bf16")])
def test_wide_head_clusters(N, d, dtype):
    """d = 512 and 1024: the CTAs of a query tile form S once as a cluster."""
    device_case(synth.Workload("guard", 1, 2, N, d, dtype, dtype == "bf16", seed=8550 + N + d),
                workspace=dtype == "fp32", expect_plan="cluster=%d" % (d // 256))


@pytest.mark.parametrize("N", [77, 300])
@pytest.mark.parametrize("d,causal", [(128, False), (64, True), (40, False)])
def test_strided_output_with_padding(N, d, causal):
    """fa_attention writing a view whose rows are 8 columns wider than d and
    whose heads are 3 rows apart: the pad columns and rows are sentinels."""
    w = synth.Workload("guard", 2, 2, N, d, "bf16", causal, seed=8600 + N + d)
    host_in, (q, k, v) = inputs(w)
    o = Guarded(w.shape, torch.bfloat16, pad=(3, 8))
    lse = Guarded(w.shape[:3], torch.float32)
    assert not o.t.is_contiguous()
    fa.fa_attention(q, k, v, o=o.t, lse=lse.t, scale=w.scale, causal=causal)
    finish(w, o, lse, host_in, "bf16")


@pytest.mark.parametrize("N", [77, 513])
@pytest.mark.parametrize("d", [64, 128])
def test_host_buffer_entry_point(N, d):
    w = synth.Workload("guard", 2, 3, N, d, "bf16", True, seed=8700 + N + d)
    host_in, (q, k, v) = inputs(w, where="pinned")
    o = Guarded(w.shape, torch.bfloat16, where="pinned")
    lse = Guarded(w.shape[:3], torch.float32, where="pinned")
    ws = torch.empty(fa.host_workspace_size(*w.shape, torch.bfloat16, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    fa.forward_host(q, k, v, o.t, lse.t, ws, scale=w.scale, causal=w.causal)
    finish(w, o, lse, host_in, "bf16")


@pytest.mark.parametrize("N", [77, 513])
def test_allocation_free_entry_point(N):
    w = synth.Workload("guard", 1, 2, N, 128, "fp32", False, seed=8800 + N)
    host_in, (q, k, v) = inputs(w)
    o = Guarded(w.shape, torch.float32)
    lse = Guarded(w.shape[:3], torch.float32)
    st = fa.load().fa_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.t.data_ptr(), lse.t.data_ptr(),
                                      w.B, w.H, w.N, w.d, w.scale, 0, fa.FA_FP32, fa.FA_FP32,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, fa.last_error()
    finish(w, o, lse, host_in, "fp32")
