"""FP8 (E4M3) drafter weights (oracle; test infrastructure).

Only tests, the smoke entry and the bench's CPU-baseline leg may import this.

Low-precision drafter weights cut the bytes a drafting round streams
([NVIDIA blog] "DFlash 如何在 NVIDIA Blackwell 上以相同的交互性提供更高的吞吐量":
decoding on Blackwell is bound by memory movement, and the platform's dense
low-precision tensor rate is quoted there).  The reading taken here:
weight-only quantisation of every projection and of the tied embedding / LM head to FP8 E4M3 with one float32 scale per output row
(per vocabulary row for the embedding), activations and accumulation as
before; the fusion projection W_fc stays bf16 (it is read once per round and
its input is the target's bf16 features).  Per row r of a bf16 matrix W:

  s_r = float32(max_k |W[r,k]|) / 448        (float32 division; 1 when the row is 0)
  q[r,k] = E4M3(float32(W[r,k]) / s_r)       (float32 division, then round to
                                              nearest even onto the E4M3 grid,
                                              saturating at +-448)
  W'[r,k] = q[r,k] * s_r                     (the weight the model then uses)

E4M3 (the OCP 8-bit floating-point format): 1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits; normal values 2^(e-7) (1 + m/8) for e = 1..15 except
the all-ones code S.1111.111 (NaN), subnormals 2^-6 * m/8; largest finite
value 448, no infinities.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_grid() -> np.ndarray:
    """All non-negative finite E4M3 values, ascending (code order 0..126)."""
    vals = []
    for code in range(127):
        e, m = code >> 3, code & 7
        vals.append(2.0 ** -6 * m / 8 if e == 0 else 2.0 ** (e - 7) * (1 + m / 8))
    return np.array(vals)


_GRID = e4m3_grid()


def round_e4m3(y: np.ndarray) -> np.ndarray:
    """Round float values to the nearest E4M3 value, ties to the even code,
    saturating at +-448 (float64 in, float64 out holding E4M3 values)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), E4M3_MAX)
    i = np.clip(np.searchsorted(_GRID, a), 1, len(_GRID) - 1)   # _GRID[i-1] < a <= _GRID[i]
    lo, hi = _GRID[i - 1], _GRID[i]
    d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((i & 1) == 0))   # tie: the even code
    r = np.where(pick_hi, hi, lo)
    r = np.where(a == 0, 0.0, r)
    return np.copysign(r, y)


def quantize_rows(w: np.ndarray):
    """Per-row E4M3 quantisation of a float matrix holding bf16 values.
    Returns (q values as float64 on the E4M3 grid, float32 scales)."""
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w32), axis=-1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (w32 / s[:, None]).astype(np.float32)
    return round_e4m3(y.astype(np.float64)), s


def _dequantize_block(w: np.ndarray) -> np.ndarray:
    q, s = quantize_rows(w)
    return q * s.astype(np.float64)[:, None]


def dequantize_rows(w: np.ndarray, rows_per_task: int = 512) -> np.ndarray:
    """The weight the FP8 drafter computes with: q * s per row (float64).
    Rows are independent, so large matrices are handled in blocks of rows on
    a thread pool; every row's arithmetic is the same either way."""
    w = np.asarray(w)
    if w.ndim != 2 or w.shape[0] <= rows_per_task:
        return _dequantize_block(w)
    from concurrent.futures import ThreadPoolExecutor
    import os
    out = np.empty(w.shape, dtype=np.float64)

    def work(r0):
        out[r0:r0 + rows_per_task] = _dequantize_block(w[r0:r0 + rows_per_task])

    with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        list(ex.map(work, range(0, w.shape[0], rows_per_task)))
    return out
