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
