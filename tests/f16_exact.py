"""Independent characterisation of IEEE binary16 rounding for the tests.

The fp16 oracle decodes with ldexp and rounds with frexp/rint.  These
helpers decode through numpy's float16 type and round by enumerating every
non-negative finite binary16 value in bit order (for non-negative IEEE
numbers the bit order is the value order), taking the nearest by comparison
with ties to the even bit pattern; the first pattern past the largest finite
value (0x7C00, +inf) stands for 2^16, the point where rounding overflows.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

_POS_BITS = np.arange(0x0000, 0x7C01, dtype=np.uint32)           # +0 ... max finite, then inf
_POS_VALS = _POS_BITS.astype(np.uint16).view(np.float16).astype(np.float64)
_POS_VALS[-1] = 2.0 ** 16


def f16_bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) & 0xFFFF).astype(np.uint16).view(np.float16) \
        .astype(np.float64)


def nearest_f16_bits(p) -> np.ndarray:
    """Round float64 values (assumed exact) to binary16 bit patterns, RNE."""
    p = np.asarray(p, dtype=np.float64)
    a = np.abs(p)
    hi = np.searchsorted(_POS_VALS, a, side="left")
    out = np.empty(a.shape, dtype=np.uint32)
    beyond = hi >= len(_POS_VALS)
    out[beyond] = 0x7C00
    ok = ~beyond
    h = hi[ok]
    av = a[ok]
    exact = _POS_VALS[h] == av
    lo = np.maximum(h - 1, 0)
    d_hi = _POS_VALS[h] - av
    d_lo = av - _POS_VALS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_BITS[h] % 2 == 0))
    out[ok] = np.where(exact | pick_hi, _POS_BITS[h], _POS_BITS[lo])
    out = out | np.where(np.signbit(p), 0x8000, 0).astype(np.uint32)
    return out.astype(np.uint16)


def nearest_f16_bits_fraction(v: Fraction) -> int:
    """The same rounding for an exact rational (exact dot products)."""
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    if a == 0:
        return 0
    h = int(np.searchsorted(_POS_VALS, float(a), side="left"))
    best = None
    for i in range(max(h - 2, 0), min(h + 2, len(_POS_VALS) - 1) + 1):
        d = abs(Fraction(float(_POS_VALS[i])) - a)
        if best is None or d < best[0] or (d == best[0] and _POS_BITS[i] % 2 == 0):
            best = (d, i)
    return int(_POS_BITS[best[1]]) | sign
