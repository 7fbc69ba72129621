"""Counter-based random numbers, reproducible on any host.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  Its i-th output for state ``s`` is
``mix(s + (i+1)*G)`` with the golden-ratio increment G and the published
two-multiply output mix.  Every number is addressed by (key, index), so a
stream can be read at any offset (e.g. the features of position p) without
generating what comes before it.

Normals use the Box-Muller transform on two uniforms (cosine branch only).
Values go float64 -> float32 (round to nearest even) -> bfloat16 (round to
nearest even) so the bit patterns are fixed by IEEE arithmetic alone.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S30 = np.uint64(30)
_S27 = np.uint64(27)
_S31 = np.uint64(31)
_S11 = np.uint64(11)
_TWO_M53 = float(2.0 ** -53)

_CHUNK = 1 << 22
_THREADS = max(1, min(16, os.cpu_count() or 1))


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> _S30)) * _M1
    z = (z ^ (z >> _S27)) * _M2
    return z ^ (z >> _S31)


def _mix_int(z: int) -> int:
    m = (1 << 64) - 1
    z &= m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def stream_key(seed: int, *ids: int) -> int:
    """Fold a seed and a tuple of integer ids into one 64-bit stream key."""
    m = (1 << 64) - 1
    k = _mix_int((seed + 0x9E3779B97F4A7C15) & m)
    for i in ids:
        k = _mix_int((k + 0x9E3779B97F4A7C15 * (int(i) + 1)) & m)
    return k


def splitmix64_bits(key: int, idx: np.ndarray) -> np.ndarray:
    """Output number ``idx`` of the SplitMix64 sequence started at ``key``."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx + np.uint64(1)) * _G
        return _mix(z)


def uniform(key: int, idx: np.ndarray) -> np.ndarray:
    """Uniform float64 in [0, 1) with 53 random bits."""
    b = splitmix64_bits(key, idx)
    return (b >> _S11).astype(np.float64) * _TWO_M53


def _normal_block(key: int, start: int, n: int) -> np.ndarray:
    i = np.arange(start, start + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        u1 = 1.0 - uniform(key, i * np.uint64(2))          # (0, 1]
        u2 = uniform(key, i * np.uint64(2) + np.uint64(1))  # [0, 1)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def normal(key: int, start: int, n: int) -> np.ndarray:
    """Standard normals number start..start+n-1 of stream ``key`` (float64)."""
    if n <= _CHUNK:
        return _normal_block(key, start, n)
    out = np.empty(n, dtype=np.float64)

    def work(off):
        m = min(_CHUNK, n - off)
        out[off:off + m] = _normal_block(key, start + off, m)

    with ThreadPoolExecutor(_THREADS) as ex:
        list(ex.map(work, range(0, n, _CHUNK)))
    return out


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 (RNE); returns uint16 bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float32, exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(key: int, start: int, n: int, scale: float = 1.0, shift: float = 0.0) -> np.ndarray:
    """shift + scale * N(0,1), rounded to bfloat16 bits, generated in chunks."""
    out = np.empty(n, dtype=np.uint16)

    def work(off):
        m = min(_CHUNK, n - off)
        z = _normal_block(key, start + off, m)
        out[off:off + m] = f64_to_bf16_bits(shift + scale * z)

    if n <= _CHUNK:
        work(0)
    else:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(work, range(0, n, _CHUNK)))
    return out
