"""The C-ABI library: it loads, exports every function include/*.h declares,
and rejects bad arguments on the host before touching the GPU."""
import glob
import os
import re

import pytest

import tiled_online_softmax_attn_gb300 as fa
from tiled_online_softmax_attn_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*[A-Za-z_][\w \*]*?\b(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load()


def test_header_declares_the_entry_points():
    assert {"fa_forward", "fa_forward_ex", "fa_check_device_error", "fa_last_error",
            "fa_version"} <= set(declared_functions())


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in fa._binding.SIGNATURES, f"{name} has no binding"


def test_library_is_built_for_sm_103a_only():
    assert fa_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_version(lib):
    assert "sm_103a" in fa.version()


@pytest.mark.parametrize("args,expect,text", [
    ((0, 16, 16, 16, 0, 1, 1, 8, 64, 1.0, 0, 0, 0), fa.FA_ERR_INVALID_ARG, "non-NULL"),
    ((16, 32, 48, 64, 0, 1, 1, 0, 64, 1.0, 0, 0, 0), fa.FA_ERR_INVALID_ARG, ">= 1"),
    ((16, 32, 48, 64, 0, 1, 1, 8, 0, 1.0, 0, 0, 0), fa.FA_ERR_INVALID_ARG, ">= 1"),
    ((16, 32, 48, 1 << 30, 0, 1, 1, 8, 64, float("inf"), 0, 0, 0), fa.FA_ERR_INVALID_ARG, "finite"),
    ((16, 32, 48, 1 << 30, 0, 1, 1, 8, 64, 1.0, 0, 7, 0), fa.FA_ERR_INVALID_ARG, "in_dtype"),
    ((16, 32, 48, 1 << 30, 0, 1, 1, 8, 64, 1.0, 0, 0, 9), fa.FA_ERR_INVALID_ARG, "o_dtype"),
    ((17, 32, 48, 1 << 30, 0, 1, 1, 8, 64, 1.0, 0, 0, 0), fa.FA_ERR_INVALID_ARG, "aligned"),
    ((16, 32, 48, 1 << 30, 0, 1, 1, 8, 4096, 1.0, 0, 0, 0), fa.FA_ERR_UNSUPPORTED, "1024"),
    ((16, 32, 48, 1 << 40, 0, 1 << 20, 1 << 10, 1 << 10, 64, 1.0, 0, 0, 0), fa.FA_ERR_UNSUPPORTED, "2^31"),
    ((1 << 30, 32, 48, 1 << 30, 0, 1, 1, 8, 64, 1.0, 0, 0, 0), fa.FA_ERR_INVALID_ARG, "overlap"),
])
def test_host_validation(lib, args, expect, text):
    assert fa.forward_raw(*args) == expect
    assert text in fa.last_error()


def test_unknown_flags_rejected(lib):
    st = fa.forward_raw(16, 32, 48, 1 << 30, 0, 1, 1, 8, 64, 1.0, 0, 0, 0, 0, 0x80)
    assert st == fa.FA_ERR_INVALID_ARG and "flag" in fa.last_error()


def test_fa_forward_requires_cuda_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros((1, 1, 4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_forward(x, x, x)


def _params(**kw):
    p = fa.FaParams()
    p.q, p.k, p.v, p.o = 1 << 40, 2 << 40, 3 << 40, 4 << 40
    p.B, p.H, p.Nq, p.Nk, p.dk, p.dv = 2, 4, 100, 70, 64, 32
    p.scale, p.causal, p.in_dtype, p.o_dtype = 0.125, 0, fa.FA_BF16, fa.FA_BF16
    for name, val in kw.items():
        if name.endswith("stride"):
            getattr(p, name)[:] = val
        else:
            setattr(p, name, val)
    return p


@pytest.mark.parametrize("kw,expect,text", [
    (dict(o_stride=[4 * 100 * 32, 32, 16]), fa.FA_ERR_INVALID_ARG, "overlap"),   # rows of 32 every 16
    (dict(q_stride=[-1, 64, 64]), fa.FA_ERR_INVALID_ARG, ">= 0"),
    (dict(o=(1 << 40) + 64), fa.FA_ERR_INVALID_ARG, "overlap"),
    (dict(Nk=0), fa.FA_ERR_INVALID_ARG, ">= 1"),
    (dict(dv=2048), fa.FA_ERR_UNSUPPORTED, "1024"),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG, "finite"),
])
def test_attention_params_validation(lib, kw, expect, text):
    import ctypes
    p = _params(**kw)
    assert lib.fa_attention(ctypes.byref(p), None, 0, None) == expect
    assert text in fa.last_error()


def test_attention_accepts_sequence_major_layout_on_the_host(lib):
    """(batch, seq, heads, dim) strides pass validation; with no GPU the call
    then fails at the launch, not before."""
    import ctypes
    B, H, Nq, Nk, dk, dv = 2, 4, 100, 70, 64, 32
    p = _params(q_stride=[Nq * H * dk, dk, H * dk], k_stride=[Nk * H * dk, dk, H * dk],
                v_stride=[Nk * H * dv, dv, H * dv], o_stride=[Nq * H * dv, dv, H * dv])
    st = lib.fa_attention(ctypes.byref(p), None, 0, None)
    assert st == fa.FA_ERR_CUDA, fa.last_error()


def test_last_error_returns_the_status_and_cuts_the_text(lib):
    import ctypes
    assert fa.forward_raw(0, 16, 16, 16, 0, 1, 1, 8, 64, 1.0, 0, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.last_status() == fa.FA_ERR_INVALID_ARG
    small = ctypes.create_string_buffer(8)
    assert lib.fa_last_error(small, len(small)) == fa.FA_ERR_INVALID_ARG
    assert len(small.value) == 7 and fa.last_error().startswith(small.value.decode())
    # a size query leaves the record alone; a later failure replaces it
    lib.fa_workspace_size(1, 1, 8, 64, 0, 0, 0)
    assert fa.last_status() == fa.FA_ERR_INVALID_ARG
    assert fa.forward_raw(16, 32, 48, 1 << 30, 0, 1, 1, 8, 4096, 1.0, 0, 0, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.last_status() == fa.FA_ERR_UNSUPPORTED and "1024" in fa.last_error()


@pytest.mark.parametrize("lse,o,expect,text", [
    ((5 << 40) + 2, 4 << 40, fa.FA_ERR_INVALID_ARG, "aligned"),     # LSE not 4-byte aligned
    (None, (1 << 40) + 64, fa.FA_ERR_INVALID_ARG, "overlap"),       # O inside Q
    (4 << 40, 4 << 40, fa.FA_ERR_INVALID_ARG, "overlap"),           # O on top of LSE
])
def test_noalloc_checks_arguments_like_the_workspace_entry_point(lib, lse, o, expect, text):
    """fa_forward_noalloc applies the rules of fa_forward_ws before anything
    else (placeholder addresses, never dereferenced: no GPU is touched)."""
    q, k, v = 1 << 40, 2 << 40, 3 << 40
    args = (q, k, v, o, lse, 1, 1, 64, 256, 0.0625, 0, fa.FA_FP32, fa.FA_FP32)
    assert lib.fa_forward_noalloc(*args, None) == expect
    assert text in fa.last_error()
    assert lib.fa_forward_ws(*args, None, 0, None) == expect


@pytest.mark.parametrize("d,dtype,path", [
    (64, fa.FA_BF16, "tensor-core"), (128, fa.FA_BF16, "tensor-core"), (8, fa.FA_BF16, "tensor-core"),
    (40, fa.FA_BF16, "tensor-core"), (120, fa.FA_BF16, "tensor-core"), (44, fa.FA_BF16, "general"),
    (136, fa.FA_BF16, "general"), (40, fa.FA_FP32, "general"), (256, fa.FA_BF16, "wide-head tensor-core bf16"),
    (128, fa.FA_FP32, "wide-head tensor-core fp32 as bf16 hi+lo")])
def test_backward_plan_picks_the_path_by_head_width(lib, d, dtype, path):
    """Host-side choice of the backward kernel: bf16 heads of a multiple of 8
    up to 128 on the tensor cores (padded below 64 and between 64 and 128),
    wider ones on the wide-head kernel, the rest on the CUDA cores."""
    n, desc = fa.backward_plan(1, 2, 300, d, dtype, True)
    assert desc == path and n >= 3


@pytest.mark.parametrize("B,H,N,d,causal,one", [
    (1, 2, 100, 64, False, True), (1, 2, 128, 64, False, True), (1, 1, 1, 128, False, True),
    (1, 2, 100, 64, True, False), (4, 32, 4096, 128, False, False)])
def test_plan_reports_single_tile_items_for_short_queries(B, H, N, d, causal, one):
    """Host-side choice of the forward's work items: unmasked problems of at
    most 128 query rows run items of one query tile whatever the device; the
    fill rule for longer queries needs the SM count, so without a GPU only the
    short-query rule shows (the GPU test checks the fill rule)."""
    import torch
    n, desc = fa.plan(B, H, N, d, torch.bfloat16, torch.bfloat16, causal)
    assert n == 1 and desc.startswith(f"tensor-core d={d}")
    if not torch.cuda.is_available():
        assert ("one query tile per item" in desc) == one, desc
