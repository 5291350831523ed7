"""Seeded synthetic inputs, shared by the tests, the bench and the oracle checks.

This module holds random-number generation only: no convolution, halo or
reduction arithmetic lives here, so the CUDA path and the CPU oracle can both
draw their inputs from it without sharing any of the method's arithmetic.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: draw ``i`` of a stream
is ``mix(key + (i + 1) * GOLDEN)``, so any element can be produced on its own
and in any order.  From the 64-bit draws:

* uniform [0, 1): the top 53 bits times 2**-53;
* normal: Box-Muller (cosine branch) on draws ``2i`` (radius, mapped to
  (0, 1]) and ``2i + 1`` (angle);
* truncated normal: a normal, resampled while ``|z| > 2`` (round ``k`` uses
  the normal at counter ``i + k * size``);
* Kaiming normal: normal with std ``sqrt(2 / fan_in)``.

Each tensor of a workload gets its own stream key ``seed * 1000 + tensor_id``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TWO53 = 2.0 ** -53
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> np.uint64:
    """Stream key of one tensor: the SplitMix64 mix of ``seed * 1000 + tensor_id``."""
    with np.errstate(over="ignore"):
        return _mix(np.array([seed * 1000 + tensor_id], dtype=np.uint64))[0]


def draws(key: np.uint64, counters: np.ndarray) -> np.ndarray:
    """Raw 64-bit draws at the given 0-based counters of stream ``key``."""
    with np.errstate(over="ignore"):
        c = counters.astype(np.uint64) + np.uint64(1)
        return _mix(key + c * GOLDEN)


def _uniform01(key, counters):
    return (draws(key, counters) >> np.uint64(11)).astype(np.float64) * _TWO53


def _normal_at(key, idx):
    z1 = draws(key, 2 * idx)
    z2 = draws(key, 2 * idx + 1)
    u1 = ((z1 >> np.uint64(11)).astype(np.float64) + 1.0) * _TWO53  # (0, 1]
    u2 = (z2 >> np.uint64(11)).astype(np.float64) * _TWO53
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def _fill(shape, fn) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float32)
    starts = list(range(0, n, _CHUNK))

    def work(s):
        e = min(n, s + _CHUNK)
        out[s:e] = fn(np.arange(s, e, dtype=np.int64), n)

    if len(starts) > 1:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    elif starts:
        work(0)
    return out.reshape(shape)


def uniform(shape, lo: float, hi: float, seed: int, tensor_id: int) -> np.ndarray:
    """float32 array, uniform on [lo, hi)."""
    key = stream_key(seed, tensor_id)
    return _fill(tuple(shape), lambda i, n: lo + (hi - lo) * _uniform01(key, i))


def normal(shape, std: float, seed: int, tensor_id: int, mean: float = 0.0) -> np.ndarray:
    """float32 array, normal(mean, std)."""
    key = stream_key(seed, tensor_id)
    return _fill(tuple(shape), lambda i, n: mean + std * _normal_at(key, i))


def trunc_normal(shape, std: float, seed: int, tensor_id: int, bound: float = 2.0) -> np.ndarray:
    """float32 array, normal(0, std) truncated to [-bound*std, bound*std] by resampling."""
    key = stream_key(seed, tensor_id)

    def fn(i, n):
        z = _normal_at(key, i)
        bad = np.abs(z) > bound
        k = 0
        while bad.any():
            k += 1
            z[bad] = _normal_at(key, i[bad] + k * n)
            bad = np.abs(z) > bound
        return std * z

    return _fill(tuple(shape), fn)


def kaiming_normal(shape, fan_in: int, seed: int, tensor_id: int) -> np.ndarray:
    """float32 array, normal(0, sqrt(2 / fan_in))."""
    return normal(shape, float(np.sqrt(2.0 / fan_in)), seed, tensor_id)


def dyadic(shape, bits: int, span: int, seed: int, tensor_id: int) -> np.ndarray:
    """float32 array of multiples of 2**-bits in [-span, span].

    Sums and products of a few such values are exact in fp32 and fp64 and in
    tf32 when ``bits`` is small, which makes exact (bit-level) checks possible.
    """
    key = stream_key(seed, tensor_id)
    levels = 2 * span * (1 << bits) + 1

    def fn(i, n):
        q = (draws(key, i) % np.uint64(levels)).astype(np.float64)
        return (q - span * (1 << bits)) / float(1 << bits)

    return _fill(tuple(shape), fn)
