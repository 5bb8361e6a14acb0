"""CPU fp64 oracle for the attention forward pass.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the bench's CPU-baseline and reference legs.  The CUDA product path
never imports, links or runs anything here, and nothing here touches the
CUDA path.

``attention_rows`` / ``attention`` wrap ``oracle.c`` (the three passes of
"Safe Softmax and the Three Passes" in "The Details of Flash Attention",
fp64); ``attention_backward`` is the gradient of that definition written
out, and ``attention_backward_sampled`` the same gradient for chosen query
rows and keys only (for problems too large for N x N weights); ``tiled_model`` holds a second, tile-by-tile restatement of the online
recurrence used only to pin the intermediate numbers of the worked example.
Row chunks run on host threads (ctypes releases the GIL during the C call).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with the host C compiler."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f = lib.oracle_attention_rows_qkv
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 6 + [
                ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            g = lib.oracle_attention_backward_head
            g.restype = ctypes.c_int
            g.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 4 + [
                ctypes.c_double, ctypes.c_int, ctypes.c_int64] + [ctypes.c_void_p] * 4
            _lib = lib
    return _lib


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def attention_rows(q, k, v, scale, causal, rows, threads=None):
    """Exact O rows and LSE for the given row ids (bh * Nq + i), in float64.

    q: [B, H, Nq, dk], k: [B, H, Nk, dk], v: [B, H, Nk, dv] float32 arrays
    holding the exact input values.  Returns (o[len(rows), dv], lse[len(rows)]).
    """
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be 4-D [B, H, N, d] arrays")
    B, H, N, d = q.shape
    Nk, dv = k.shape[2], v.shape[3]
    if k.shape != (B, H, Nk, d) or v.shape != (B, H, Nk, dv):
        raise ValueError("k must be [B, H, Nk, dk] and v [B, H, Nk, dv] with q's B, H, dk")
    rows = np.ascontiguousarray(rows, dtype=np.int64).ravel()
    o = np.empty((rows.size, dv), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    if rows.size == 0:
        return o, lse
    lib = _load()
    threads = threads or default_threads()
    nchunks = min(rows.size, max(1, threads * 4))
    bounds = np.linspace(0, rows.size, nchunks + 1).astype(np.int64)

    def run(c):
        lo, hi = int(bounds[c]), int(bounds[c + 1])
        if hi <= lo:
            return 0
        work = np.empty(Nk, dtype=np.float64)
        return lib.oracle_attention_rows_qkv(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, N, Nk, d, dv,
            float(scale), int(bool(causal)), rows[lo:].ctypes.data, hi - lo,
            o[lo:].ctypes.data, lse[lo:].ctypes.data, work.ctypes.data)

    if threads == 1 or nchunks == 1:
        codes = [run(c) for c in range(nchunks)]
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            codes = list(ex.map(run, range(nchunks)))
    bad = [c for c in codes if c != 0]
    if bad:
        raise RuntimeError(f"oracle_attention_rows failed with code {bad[0]}")
    return o, lse


def attention(q, k, v, scale, causal=False, threads=None):
    """Exact O [B, H, Nq, dv] and LSE [B, H, Nq] for every row, in float64."""
    B, H, N, _ = np.shape(q)
    dv = np.shape(v)[3]
    rows = np.arange(B * H * N, dtype=np.int64)
    o, lse = attention_rows(q, k, v, scale, causal, rows, threads)
    return o.reshape(B, H, N, dv), lse.reshape(B, H, N)


def attention_backward(q, k, v, dout, scale, causal=False, threads=None):
    """Gradients (dq, dk, dv) of L = sum(O * dout) for the forward pass on
    q, k, v [B, H, N, d] (float32 arrays of the exact input values), float64.
    Heads run on host threads; each materialises its N x N weights."""
    q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
    if q.ndim != 4 or not (q.shape == k.shape == v.shape == dout.shape):
        raise ValueError("q, k, v, dout must be [B, H, N, d] arrays of one shape")
    B, H, N, d = q.shape
    dq, dk, dv = (np.empty((B * H, N, d), dtype=np.float64) for _ in range(3))
    lib = _load()

    def run(bh):
        work = np.empty(N * N, dtype=np.float64)
        return lib.oracle_attention_backward_head(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, B, H, N, d,
            float(scale), int(bool(causal)), bh, dq[bh].ctypes.data, dk[bh].ctypes.data,
            dv[bh].ctypes.data, work.ctypes.data)

    threads = threads or default_threads()
    with ThreadPoolExecutor(max_workers=max(1, min(threads, B * H))) as ex:
        codes = list(ex.map(run, range(B * H)))
    if any(codes):
        raise RuntimeError("oracle_attention_backward_head failed")
    shape = (B, H, N, d)
    return dq.reshape(shape), dk.reshape(shape), dv.reshape(shape)


def attention_backward_sampled(q, k, v, dout, scale, causal, rows, keys, threads=None):
    """Gradients of chosen query rows (dQ) and chosen keys (dK, dV), float64.

    The definition of ``attention_backward`` evaluated for a subset: with
    S_ij = scale * q_i . k_j, the row statistics LSE_i and O_i of the forward
    oracle, P_ij = exp(S_ij - LSE_i) (0 for a masked pair), dP_ij = dO_i . v_j
    and delta_i = dO_i . O_i (= sum_j P_ij dP_ij):

        dQ_i = scale * sum_j P_ij (dP_ij - delta_i) k_j
        dK_j = scale * sum_i P_ij (dP_ij - delta_i) q_i
        dV_j = sum_i P_ij dO_i

    rows / keys hold flat ids bh * N + i.  A key's gradients sum over every
    query of its head, so each head with a chosen key gets the forward oracle
    over all of its rows.  Returns (dq[len(rows), d], dk[len(keys), d],
    dv[len(keys), d]).
    """
    q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
    if q.ndim != 4 or not (q.shape == k.shape == v.shape == dout.shape):
        raise ValueError("q, k, v, dout must be [B, H, N, d] arrays of one shape")
    B, H, N, d = q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64).ravel()
    keys = np.ascontiguousarray(keys, dtype=np.int64).ravel()
    if np.any((rows < 0) | (rows >= B * H * N)) or np.any((keys < 0) | (keys >= B * H * N)):
        raise ValueError("row or key id out of range")
    qf, kf, vf, gf = (x.reshape(B * H, N, d).astype(np.float64) for x in (q, k, v, dout))
    dq = np.empty((rows.size, d))
    dk = np.empty((keys.size, d))
    dv = np.empty((keys.size, d))
    # query rows: their own statistics suffice
    if rows.size:
        o_r, lse_r = attention_rows(q, k, v, scale, causal, rows, threads)
        for n, r in enumerate(rows):
            bh, i = divmod(int(r), N)
            nk = i + 1 if causal else N
            s = scale * (kf[bh, :nk] @ qf[bh, i])
            p = np.exp(s - lse_r[n])
            dp = vf[bh, :nk] @ gf[bh, i]
            delta = float(gf[bh, i] @ o_r[n])
            dq[n] = scale * ((p * (dp - delta)) @ kf[bh, :nk])
    # keys: every query of the head
    for bh in np.unique(keys // N):
        sel = np.nonzero(keys // N == bh)[0]
        js = keys[sel] - bh * N
        o_h, lse_h = attention_rows(q, k, v, scale, causal, np.arange(N, dtype=np.int64) + bh * N, threads)
        delta = np.einsum("id,id->i", gf[bh], o_h)
        s = scale * (qf[bh] @ kf[bh, js].T)                      # [N queries, chosen keys]
        p = np.exp(s - lse_h[:, None])
        if causal:
            p = np.where(np.arange(N)[:, None] >= js[None, :], p, 0.0)
        dp = gf[bh] @ vf[bh, js].T
        ds = p * (dp - delta[:, None])
        dk[sel] = scale * (ds.T @ qf[bh])
        dv[sel] = p.T @ gf[bh]
    return dq, dk, dv
