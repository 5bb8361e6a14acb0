"""ctypes binding of the C ABI in include/fa.h.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of libfa_gb300.so.  There is no fallback -- if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA",
                4: "FA_ERR_TIMEOUT"}

FA_BF16 = 0
FA_FP32 = 1
FA_FLAG_GENERAL_PATH = 0x1
FA_FLAG_TEST_SKIP_KV_LOAD = 0x100

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa_gb300.so")

_I64 = ctypes.c_int64
_P = ctypes.c_void_p


class FaParams(ctypes.Structure):
    """struct fa_params of include/fa.h."""
    _fields_ = [("q", _P), ("k", _P), ("v", _P), ("o", _P), ("lse", _P),
                ("B", _I64), ("H", _I64), ("Nq", _I64), ("Nk", _I64), ("dk", _I64), ("dv", _I64),
                ("q_stride", _I64 * 3), ("k_stride", _I64 * 3), ("v_stride", _I64 * 3),
                ("o_stride", _I64 * 3), ("scale", ctypes.c_float), ("causal", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("o_dtype", ctypes.c_int)]


# name -> (restype, argtypes) for every function include/fa.h declares
SIGNATURES = {
    "fa_forward": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]),
    "fa_forward_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, ctypes.c_uint32]),
    "fa_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "fa_plan": (ctypes.c_int, [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_size_t, ctypes.c_char_p, ctypes.c_size_t]),
    "fa_forward_ws": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "fa_host_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int]),
    "fa_forward_host": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "fa_attention": (ctypes.c_int, [ctypes.POINTER(FaParams), _P, ctypes.c_size_t, _P]),
    "fa_attention_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(FaParams)]),
    "fa_backward_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64, _I64]),
    "fa_backward_workspace_size_ex": (ctypes.c_size_t, [_I64, _I64, _I64, _I64, ctypes.c_int]),
    "fa_backward_plan": (ctypes.c_int, [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_size_t,
                                        ctypes.c_char_p, ctypes.c_size_t]),
    "fa_backward": (ctypes.c_int, [_P] * 9 + [_I64, _I64, _I64, _I64, ctypes.c_float, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "fa_forward_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]),
    "fa_check_device_error": (ctypes.c_int, [_P]),
    "fa_last_error": (ctypes.c_int, [ctypes.c_char_p, ctypes.c_size_t]),
    "fa_version": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load(path: str | None = None):
    """Load libfa_gb300.so (built by ``build()``) and bind its symbols."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise FileNotFoundError(
                f"{p} is missing: build the CUDA library first (__graft_entry__.build())")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        if path is None:
            _lib = lib
        return lib


def last_error() -> str:
    """Text of the last failure of an fa_* call on this host thread ("" if it succeeded)."""
    buf = ctypes.create_string_buffer(1024)
    load().fa_last_error(buf, len(buf))
    return buf.value.decode()


def last_status() -> int:
    """fa_status the last fa_* call on this host thread returned."""
    return int(load().fa_last_error(None, 0))


def version() -> str:
    return load().fa_version().decode()


def check(status: int) -> None:
    if status != FA_OK:
        raise FAError(status, last_error())


def forward_raw(q, k, v, o, lse, B, H, N, d, scale, causal, in_dtype, o_dtype, stream=0, flags=0) -> int:
    """Direct call with integer pointers; returns the fa_status."""
    lib = load()
    return lib.fa_forward_ex(q, k, v, o, lse, B, H, N, d, scale, int(bool(causal)), in_dtype,
                             o_dtype, stream, flags)


def check_device_error(stream=0) -> int:
    return load().fa_check_device_error(stream)


def _dtype_code(t) -> int:
    import torch
    if t == torch.bfloat16:
        return FA_BF16
    if t == torch.float32:
        return FA_FP32
    raise TypeError(f"unsupported dtype {t}")


def workspace_size(B, H, N, d, in_dtype, o_dtype, causal=False) -> int:
    """Device workspace bytes fa_forward_ws can use (dtypes: torch dtypes or FA_* codes)."""
    ic = in_dtype if isinstance(in_dtype, int) else _dtype_code(in_dtype)
    oc = o_dtype if isinstance(o_dtype, int) else _dtype_code(o_dtype)
    return int(load().fa_workspace_size(B, H, N, d, ic, oc, int(bool(causal))))


def plan(B, H, N, d, in_dtype, o_dtype, causal=False, workspace_bytes=0):
    """(kernel launches per call, description) of the path fa_forward_ws takes."""
    ic = in_dtype if isinstance(in_dtype, int) else _dtype_code(in_dtype)
    oc = o_dtype if isinstance(o_dtype, int) else _dtype_code(o_dtype)
    buf = ctypes.create_string_buffer(160)
    n = load().fa_plan(B, H, N, d, ic, oc, int(bool(causal)), workspace_bytes, buf, len(buf))
    return int(n), buf.value.decode()


def fa_forward(q, k, v, o=None, lse=None, scale=None, causal=False, o_dtype=None,
               return_lse=True, stream=None, flags=0, workspace=None):
    """O = softmax(q k^T * scale) v on [B, H, N, d] CUDA tensors.

    Returns (o, lse); ``lse`` is None when ``return_lse`` is False and no
    buffer was passed.  ``o``/``lse`` may be given to write into existing
    buffers.  ``scale`` defaults to 1/sqrt(d).  The call is asynchronous on
    ``stream`` (default: torch's current stream).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor [B, H, N, d]")
    if q.shape != k.shape or q.shape != v.shape or q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k, v must share shape and dtype")
    B, H, N, d = q.shape
    in_code = _dtype_code(q.dtype)
    if o is None:
        o = torch.empty(q.shape, dtype=o_dtype or q.dtype, device=q.device)
    elif not o.is_contiguous() or o.shape != q.shape:
        raise ValueError("o must be contiguous with q's shape")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.shape != (B, H, N)):
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            lse.data_ptr() if lse is not None else None, B, H, N, d, float(scale),
            int(bool(causal)), in_code, _dtype_code(o.dtype))
    if workspace is not None:
        if flags:
            raise ValueError("flags are not available together with a workspace")
        if not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        st = load().fa_forward_ws(*args, workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), stream)
    else:
        st = forward_raw(*args, stream, flags)
    check(st)
    return o, lse


def host_workspace_size(B, H, N, d, in_dtype, o_dtype) -> int:
    """Device workspace bytes fa_forward_host needs (dtypes: torch dtypes or FA_* codes)."""
    ic = in_dtype if isinstance(in_dtype, int) else _dtype_code(in_dtype)
    oc = o_dtype if isinstance(o_dtype, int) else _dtype_code(o_dtype)
    return int(load().fa_host_workspace_size(B, H, N, d, ic, oc))


def forward_host(q, k, v, o, lse, workspace, scale=None, causal=False, stream=None):
    """fa_forward_host on CPU tensors (pinned for overlap); ``workspace`` is a
    CUDA uint8 tensor of at least host_workspace_size bytes.  Synchronous."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D host tensor")
    if q.shape != k.shape or q.shape != v.shape or q.shape != o.shape:
        raise ValueError("q, k, v, o must share one shape")
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    if lse is not None and (lse.is_cuda or lse.dtype != torch.float32 or lse.shape != (B, H, N)):
        raise ValueError("lse must be a float32 [B, H, N] host tensor")
    st = load().fa_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr() if lse is not None else None, B, H, N, d,
                                float(scale), int(bool(causal)), _dtype_code(q.dtype),
                                _dtype_code(o.dtype), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), stream)
    check(st)
    return o, lse


def _fa_params(q, k, v, o, lse, scale, causal):
    B, H, Nq, dk = q.shape
    Nk, dv = k.shape[2], v.shape[3]
    prm = FaParams()
    prm.q, prm.k, prm.v, prm.o = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr()
    prm.lse = lse.data_ptr() if lse is not None else None
    prm.B, prm.H, prm.Nq, prm.Nk, prm.dk, prm.dv = B, H, Nq, Nk, dk, dv
    for name, t in (("q_stride", q), ("k_stride", k), ("v_stride", v), ("o_stride", o)):
        getattr(prm, name)[:] = list(t.stride()[:3])
    prm.scale, prm.causal = float(scale), int(bool(causal))
    prm.in_dtype, prm.o_dtype = _dtype_code(q.dtype), _dtype_code(o.dtype)
    return prm


def attention_workspace_size(q, k, v, o=None, causal=False, o_dtype=None) -> int:
    """fa_attention_workspace_size: device workspace bytes that let
    fa_attention run these tensors at full parallelism (o: the output view,
    or a contiguous [B, H, Nq, dv] tensor of o_dtype when None)."""
    prm = _fa_params(q, k, v, q if o is None else o, None, 1.0, causal)  # the size query reads no pointer
    if o is None:
        B, H, Nq, _ = q.shape
        dv = v.shape[3]
        prm.o_stride[:] = [H * Nq * dv, Nq * dv, dv]
        prm.o_dtype = _dtype_code(o_dtype or q.dtype)
    return int(load().fa_attention_workspace_size(ctypes.byref(prm)))


def fa_attention(q, k, v, o=None, lse=None, scale=None, causal=False, o_dtype=None,
                 return_lse=True, workspace=None, stream=None):
    """Attention on [B, H, Nq, dk] / [B, H, Nk, dk] / [B, H, Nk, dv] CUDA tensors
    with any strides (the last dimension contiguous), e.g. transposed views of
    (batch, seq, heads, dim) tensors.  O defaults to a contiguous
    [B, H, Nq, dv] tensor; an existing (possibly strided) view may be passed."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or t.dim() != 4 or t.stride(-1) != 1:
            raise ValueError(f"{name} must be a 4-D CUDA tensor whose last dimension is contiguous")
    B, H, Nq, dk = q.shape
    Nk, dv = k.shape[2], v.shape[3]
    if k.shape != (B, H, Nk, dk) or v.shape != (B, H, Nk, dv) or q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("k must be [B, H, Nk, dk] and v [B, H, Nk, dv], one dtype")
    if o is None:
        o = torch.empty((B, H, Nq, dv), dtype=o_dtype or q.dtype, device=q.device)
    elif o.shape != (B, H, Nq, dv) or o.stride(-1) != 1:
        raise ValueError("o must be [B, H, Nq, dv] with a contiguous last dimension")
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.shape != (B, H, Nq)):
        raise ValueError("lse must be a contiguous float32 [B, H, Nq] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    prm = _fa_params(q, k, v, o, lse, scale, causal)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(load().fa_attention(ctypes.byref(prm), ws_ptr, ws_bytes, stream))
    return o, lse


def fa_backward(q, k, v, o, dout, lse, scale=None, causal=False, grad_dtype=None, dq=None, dk=None,
                dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of the forward pass that produced (o, lse) from
    q, k, v, given dout = dL/dO; contiguous [B, H, N, d] CUDA tensors."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if not t.is_cuda or not t.is_contiguous() or t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor like q")
    B, H, N, d = q.shape
    gdt = grad_dtype or q.dtype
    dq = torch.empty(q.shape, dtype=gdt, device=q.device) if dq is None else dq
    dk = torch.empty(q.shape, dtype=gdt, device=q.device) if dk is None else dk
    dv = torch.empty(q.shape, dtype=gdt, device=q.device) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(backward_workspace_size(B, H, N, d, q.dtype), dtype=torch.uint8, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    st = load().fa_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                            float(scale), int(bool(causal)), _dtype_code(q.dtype), _dtype_code(gdt),
                            workspace.data_ptr(), workspace.numel() * workspace.element_size(), stream)
    check(st)
    return dq, dk, dv


def backward_workspace_size(B, H, N, d, in_dtype) -> int:
    """Workspace bytes that let fa_backward run on the tensor cores where it can
    (dtype: a torch dtype or an FA_* code)."""
    ic = in_dtype if isinstance(in_dtype, int) else _dtype_code(in_dtype)
    return int(load().fa_backward_workspace_size_ex(B, H, N, d, ic))


def backward_plan(B, H, N, d, in_dtype, causal=False, workspace_bytes=None):
    """(kernel launches per call, description) of the path fa_backward takes
    (workspace_bytes defaults to backward_workspace_size)."""
    ic = in_dtype if isinstance(in_dtype, int) else _dtype_code(in_dtype)
    if workspace_bytes is None:
        workspace_bytes = backward_workspace_size(B, H, N, d, ic)
    buf = ctypes.create_string_buffer(96)
    n = load().fa_backward_plan(B, H, N, d, ic, int(bool(causal)), workspace_bytes, buf, len(buf))
    return int(n), buf.value.decode()
