"""FP8 (e4m3) KV-cache codec — TEST INFRASTRUCTURE (CPU oracle).

e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
S.1111.111 is NaN; largest finite 448, smallest normal 2^-6, smallest
subnormal 2^-9. A cache value is code * scale, with one scale per KV head for K
and one for V. Quantising takes y = x / scale in IEEE float32 (correctly
rounded), then rounds y to the nearest e4m3 value, ties to even, saturating
to +-448.
"""
from __future__ import annotations

import numpy as np


def e4m3_table() -> np.ndarray:
    """Value of each of the 256 codes (float64; NaN for the two NaN codes)."""
    out = np.empty(256, dtype=np.float64)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            v = np.nan
        elif e == 0:
            v = 2.0 ** -6 * (m / 8.0)
        else:
            v = 2.0 ** (e - 7) * (1.0 + m / 8.0)
        out[c] = -v if s else v
    return out


_TABLE = e4m3_table()
_POS = _TABLE[:127]          # codes 0..126: the non-negative finite values, increasing


def quantize(x, scale) -> np.ndarray:
    """Codes (uint8) of x / scale: float32 division, nearest e4m3, ties to even,
    saturating. x [..., H, d]; scale [H] (broadcast over the last axis)."""
    y = (np.asarray(x, dtype=np.float32) / np.asarray(scale, dtype=np.float32)[..., :, None]).astype(np.float64)
    a = np.minimum(np.abs(y), 448.0)
    # nearest of the increasing finite values, ties to the even code
    hi = np.searchsorted(_POS, a, side="left")
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _POS[lo], _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == _POS[hi], hi, code).astype(np.uint8)
    sign = (np.signbit(y)).astype(np.uint8) << 7
    out = code | sign
    return np.where(np.isnan(y), np.uint8(0x7F), out).astype(np.uint8)


def dequantize(codes, scale) -> np.ndarray:
    """float64 values code * scale; codes [..., H, d], scale [H]."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)] * np.asarray(scale, dtype=np.float64)[..., :, None]
