"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the CPU oracle side and the CUDA side of the tests
and the bench; it holds no attention arithmetic, only random numbers.

Generator (counter based, so any element can be produced on its own and the
values do not depend on chunking, on numpy's or torch's RNG, or on the host):

* ``bits(stream, c)`` is SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014): the output of the 64-bit
  finaliser ``mix`` applied to ``key(stream) + (c + 1) * GOLDEN`` where
  ``key(stream) = mix((stream + 1) * GOLDEN)``.
* ``uniform(stream, c) = ((bits >> 11) + 1) * 2**-53``, in (0, 1].
* element ``e`` of a standard normal stream is the Box-Muller transform
  ``sqrt(-2 ln u1) * cos(2 pi u2)`` of ``u1 = uniform(stream, 2e)`` and
  ``u2 = uniform(stream, 2e + 1)``, computed in float64.
* bf16 inputs are that float64 value rounded to float32 and then to bf16 with
  round-to-nearest-even; they are handed around as float32 arrays holding
  bf16-exact values, so converting them to a bf16 tensor is exact.
* Q, K and V of a workload with seed ``s`` use streams ``3s``, ``3s+1`` and
  ``3s+2``.

The workloads are the five shapes the pages' discussion leads to (a tiny
case, the single-head d=1024 fp32 shape of the eight-kernel CUDA walkthrough
in "The Details of Flash Attention", a multi-head training shape, a causal
long-context shape and a very long sequence with peaked scores).
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S30 = np.uint64(30)
_S27 = np.uint64(27)
_S31 = np.uint64(31)
_S11 = np.uint64(11)
_ONE = np.uint64(1)

CHUNK = 1 << 20


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> _S30)) * _M1
    z = (z ^ (z >> _S27)) * _M2
    return z ^ (z >> _S31)


def key(stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = np.array([(stream + 1) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64) * GOLDEN
        return _mix(z)[0]


def bits(stream: int, counters: np.ndarray) -> np.ndarray:
    """SplitMix64 outputs for the given counters of one stream."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key(stream) + (c + _ONE) * GOLDEN)


def uniform(stream: int, counters: np.ndarray) -> np.ndarray:
    b = bits(stream, counters)
    return ((b >> _S11) + _ONE).astype(np.float64) * (2.0 ** -53)


def normal(stream: int, n: int, start: int = 0) -> np.ndarray:
    """Elements ``start .. start+n-1`` of a standard normal stream, float64."""
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, CHUNK):
        hi = min(n, lo + CHUNK)
        e = np.arange(start + lo, start + hi, dtype=np.uint64)
        u1 = uniform(stream, e * np.uint64(2))
        u2 = uniform(stream, e * np.uint64(2) + _ONE)
        out[lo:hi] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return out


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 out."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & _ONE)) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).reshape(f.shape)


def tensor(stream: int, shape, dtype: str, mult: float = 1.0) -> np.ndarray:
    """A float32 array of the given shape drawn from one stream.

    ``dtype`` is "bf16" (values rounded to bf16) or "fp32".  ``mult`` is
    applied after rounding and must then be a power of two so that the
    product stays exact.
    """
    if dtype not in ("bf16", "fp32"):
        raise ValueError(f"unknown dtype {dtype!r}")
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)

    def fill(lo):
        hi = min(n, lo + CHUNK)
        x = normal(stream, hi - lo, lo).astype(np.float32)
        out[lo:hi] = round_to_bf16(x) if dtype == "bf16" else x

    starts = range(0, n, CHUNK)
    if len(starts) > 1:
        # numpy releases the GIL inside these array operations
        with ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 1)) as ex:
            list(ex.map(fill, starts))
    elif n:
        fill(0)
    if mult != 1.0:
        m, e = math.frexp(mult)
        if m != 0.5:
            raise ValueError("mult must be a power of two")
        out *= np.float32(mult)
    return out.reshape(shape)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "bf16" or "fp32": input (and output) element type
    causal: bool
    seed: int
    qk_mult: float = 1.0  # Q and K are multiplied by this after rounding

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def shape(self):
        return (self.B, self.H, self.N, self.d)

    @property
    def flops(self) -> float:
        """Two matmuls of 2*N*N*d each per head; half of them under a causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def elt_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def bytes(self) -> float:
        """Read Q, K, V once, write O and the fp32 LSE once."""
        bh_n = self.B * self.H * self.N
        return 4.0 * bh_n * self.d * self.elt_bytes + 4.0 * bh_n

    def inputs(self):
        s = self.seed
        q = tensor(3 * s + 0, self.shape, self.dtype, self.qk_mult)
        k = tensor(3 * s + 1, self.shape, self.dtype, self.qk_mult)
        v = tensor(3 * s + 2, self.shape, self.dtype)
        return q, k, v

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 256, 64, "bf16", False, 1),
    "large_d": Workload("large_d", 1, 1, 1024, 1024, "fp32", False, 2),
    "multihead": Workload("multihead", 4, 32, 4096, 128, "bf16", False, 3),
    "causal": Workload("causal", 1, 32, 16384, 128, "bf16", True, 4),
    "peaked": Workload("peaked", 1, 8, 65536, 64, "bf16", False, 5, qk_mult=4.0),
}
