"""8-bit (E4M3) cache storage for the float64 oracle.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module.

The reading note "Low-Rank Key Value Attention" counts cache payload as
elements times element size (section 4, equation 9) and asks that the width
a kernel actually allocates be recorded separately from the logical one.
Storing the cache in 8 bits halves that payload.  The format is not on the
pages; it is the OCP 8-bit floating point "E4M3" encoding, written here from
its definition:
  * one sign bit, four exponent bits (bias 7), three mantissa bits;
  * exponent field 0 holds zero and the subnormals m * 2^-9;
  * no infinities: exponent 15 with mantissa 7 is NaN, so the largest finite
    magnitude is 1.75 * 2^8 = 448.
Storage rule (a reading, stated with the library's other readings): a pool
with scale s stores the code of x / s, rounded to the nearest representable
value with ties to the even mantissa; finite values beyond 448 saturate to
+-448; the stored value is decode(code) * s.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def e4m3_decode(codes):
    """Value of each 8-bit code (float64; NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e.astype(np.float64) - 7))
    mag = np.where((e == 15) & (c & 0x7 == 7), np.nan, mag)
    return sign * mag


# codes 0x00 .. 0x7E in order are the non-negative finite values, ascending
_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(x):
    """Nearest code (ties to the even mantissa, saturating at +-448)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)  # saturate (infinities included)
    hi = np.clip(np.searchsorted(_POS, a), 1, 0x7E)  # first value >= a
    lo = hi - 1
    d_lo, d_hi = a - _POS[lo], _POS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(E4M3_NAN), code).astype(np.uint8)


def quantize(x, scale):
    """Stored codes of the values x in a pool with this scale."""
    return e4m3_encode(np.asarray(x, np.float64) / scale)


def dequantize(codes, scale):
    """Values a pool with this scale holds."""
    return e4m3_decode(codes) * scale
