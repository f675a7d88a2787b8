"""Seeded synthetic inputs, shared by the tests, the benchmark and the oracle's
callers.  This module holds none of the MoE method's arithmetic: it only
turns (seed, tensor tag, element index) into numbers.

Generator (counter based, so any slice of any tensor can be produced on its
own, on the host here or on the device by ``moe_synth_normal``):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; constants as published by Vigna): the stream key
  is ``mix64(seed * GAMMA + tag)`` and element ``i`` of the stream is
  ``u = mix64(key + (i + 1) * GAMMA)`` (all arithmetic mod 2**64).
* Box-Muller (1958), cosine branch only: ``u1 = (u >> 32 + 1) / 2**32`` in
  (0, 1], ``u2 = (u & 0xffffffff) / 2**32`` in [0, 1),
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)``, evaluated in float64.
* The tensor value is ``std * z`` rounded to fp32 (round to nearest even);
  bf16 tensors round that fp32 value again to bf16 (round to nearest even).
"""

from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1
TWO_PI = 6.283185307179586  # the float64 nearest to 2*pi

# One tag per tensor role, so every tensor is an independent stream.
TAG = dict(x=1, w_r=2, gate_bias=3, sel_bias=4, w1=5, b1=6, w2=7, b2=8,
           w1_shared=9, w2_shared=10, dy=11, zipf_rank=12)

_CHUNK = 1 << 16          # elements per work item (fits in L2)
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = _cf.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def mix64_int(z: int) -> int:
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def stream_key(seed: int, tag: int) -> int:
    return mix64_int((seed * GAMMA + tag) & _MASK)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(_M1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, tag: int, start: int, n: int) -> np.ndarray:
    """Elements [start, start+n) of the stream as uint64."""
    key = np.uint64(stream_key(seed, tag))
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + i * np.uint64(GAMMA))


def normal_f64(seed: int, tag: int, start: int, n: int) -> np.ndarray:
    u = raw_u64(seed, tag, start, n)
    u1 = ((u >> np.uint64(32)).astype(np.float64) + 1.0) * (2.0 ** -32)
    u2 = (u & np.uint64(0xFFFFFFFF)).astype(np.float64) * (2.0 ** -32)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(TWO_PI * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and return the 16-bit patterns."""
    b = np.ascontiguousarray(a, np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal(shape, std: float, seed: int, tag: int, dtype: str = "f32", start: int = 0) -> np.ndarray:
    """A seeded N(0, std^2) tensor of ``shape``.  dtype "f32" returns float32;
    "bf16" returns the bf16 values widened exactly to float32 (use
    ``f32_to_bf16_bits`` for the raw bits).  ``start`` offsets the element
    counter, so a slice of a larger tensor can be generated on its own."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)

    def work(s):
        m = min(_CHUNK, n - s)
        v = (np.float64(std) * normal_f64(seed, tag, start + s, m)).astype(np.float32)
        if dtype == "bf16":
            v = bf16_bits_to_f32(f32_to_bf16_bits(v))
        out[s:s + m] = v

    if n <= 4 * _CHUNK:
        for s in range(0, n, _CHUNK):
            work(s)
    else:  # numpy releases the GIL in these ufuncs: chunks run in parallel
        list(_pool().map(work, range(0, n, _CHUNK)))
    return out.reshape(shape)


def rows(shape_full, row_ids, std: float, seed: int, tag: int, dtype: str = "f32") -> np.ndarray:
    """Selected rows (leading index) of a seeded 2-D-or-more tensor."""
    row_len = int(np.prod(shape_full[1:]))
    out = np.empty((len(row_ids), row_len), np.float32)
    for j, r in enumerate(row_ids):
        out[j] = normal((row_len,), std, seed, tag, dtype, start=int(r) * row_len)
    return out.reshape((len(row_ids),) + tuple(shape_full[1:]))


def random_ranks(n: int, seed: int, tag: int = TAG["zipf_rank"]) -> np.ndarray:
    """A seeded random ranking 1..n of n items (rank of item i)."""
    u = raw_u64(seed, tag, 0, n)
    order = np.argsort(u, kind="stable")
    ranks = np.empty(n, np.int64)
    ranks[order] = np.arange(1, n + 1)
    return ranks
