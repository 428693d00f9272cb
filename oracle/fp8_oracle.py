"""CPU oracle of the fp8 (E4M3) projection variant: quantisation and the scaled
matrix-vector products of a decode step's projections.

TEST INFRASTRUCTURE. Only the tests and the benchmark may import this module;
the product path never calls it and shares no code with it.

The pages name fp8 only as a current topic of the nanochat project
(一天一个开源项目（第22篇）：nanochat, m.alixixi.com, section 项目简介, the
"版本" bullet); they define no number format or scaling. The readings used here,
each a plain choice:

* the format is E4M3 without infinities: 1 sign bit, 4 exponent bits with bias 7,
  3 mantissa bits; normal values (1 + m/8) * 2^(e-7) for e = 1..15 except the
  all-ones pattern (NaN), so the largest finite value is 1.75 * 2^8 = 448; the
  subnormals (m/8) * 2^-6 for e = 0;
* rounding to the nearest representable value, ties to the even mantissa; values
  past 448 in magnitude saturate to +-448;
* a weight matrix is scaled per output row: s_r = max_k |W[r, k]| / 448 (1 for a
  zero row), codes q(W[r, k] / s_r);
* an activation vector is scaled per token over its whole length the same way;
* y[t, r] = s_r * s_t * sum_k q_W[r, k] * q_x[t, k].

The scale and the scaled value decide an integer (the code). They are computed
in float32, the precision the kernel uses, so that both sides take the same
decision. The dot products are exact (float64).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_grid():
    """All non-negative finite E4M3 values, ascending, from the format definition."""
    vals = [m / 8.0 * 2.0 ** -6 for m in range(8)]          # e = 0: subnormals (and 0)
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue                                     # all ones: NaN
            vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_GRID = e4m3_grid()
# mantissa parity of each grid value (ties go to the even one): index within its
# binade of 8 (subnormals: their m)
_EVEN = np.array([(i % 8) % 2 == 0 for i in range(len(_GRID))])


def quantize_e4m3(v):
    """Nearest E4M3 value of each element (ties to even mantissa, saturating at
    +-448), returned as float64. NaN stays NaN."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    a_sat = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_GRID, a_sat, side="left")          # first grid value >= a
    hi = np.minimum(hi, len(_GRID) - 1)
    lo = np.maximum(hi - 1, 0)
    g_hi, g_lo = _GRID[hi], _GRID[lo]
    d_hi, d_lo = g_hi - a_sat, a_sat - g_lo
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & _EVEN[hi] & (hi != lo))
    exact = g_hi == a_sat
    q = np.where(exact | pick_hi, g_hi, g_lo)
    q = np.where(np.isnan(v), np.nan, q)
    return np.copysign(q, v)


def row_scales(w):
    """Per-row scale max|w| / 448 in float32 (1 for a zero row)."""
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w32), axis=-1)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def quantize_rows(w):
    """(codes as float64 values, float32 scales) of a matrix scaled per row."""
    w32 = np.asarray(w, dtype=np.float32)
    s = row_scales(w32)
    scaled = (w32 / s[:, None]).astype(np.float32)   # float32 division, as the kernel
    return quantize_e4m3(scaled), s


def gemv_e4m3(wq, w_scale, x):
    """y[t, r] = s_r * s_t * sum_k wq[r, k] * q(x[t, k] / s_t), with the activations
    quantised per token (row_scales / quantize_rows applied to x)."""
    xq, x_scale = quantize_rows(x)
    acc = np.asarray(xq, np.float64) @ np.asarray(wq, np.float64).T      # [T, R]
    return acc * np.asarray(x_scale, np.float64)[:, None] * np.asarray(w_scale, np.float64)[None, :]
