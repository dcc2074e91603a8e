"""Independent characterisation of bf16 rounding for the tests.

The oracle rounds with frexp/rint/ldexp.  These helpers instead enumerate
every non-negative finite bf16 value in bit order (for non-negative IEEE
numbers the bit pattern order is the value order) and pick the nearest value
by comparison, ties to the even bit pattern, with the first pattern past the
largest finite one (0x7F80, +inf) standing for 2^128.  That is the IEEE-754
definition of round-to-nearest-even, reached by a different route.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

_POS_BITS = np.arange(0x0000, 0x7F81, dtype=np.uint32)          # +0 ... max finite, then inf
_POS_VALS = (_POS_BITS << 16).view(np.float32).astype(np.float64)
_POS_VALS[-1] = 2.0 ** 128                                          # stand-in for the overflow point


def bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint32) & 0xFFFF
    return (b << 16).view(np.float32).astype(np.float64)


def nearest_bf16_bits(p) -> np.ndarray:
    """Round float64 values (assumed exact) to bf16 bit patterns, RNE."""
    p = np.asarray(p, dtype=np.float64)
    a = np.abs(p)
    hi = np.searchsorted(_POS_VALS, a, side="left")
    out = np.empty(a.shape, dtype=np.uint32)
    beyond = hi >= len(_POS_VALS)
    out[beyond] = 0x7F80
    ok = ~beyond
    h = hi[ok]
    av = a[ok]
    exact = _POS_VALS[h] == av
    lo = np.maximum(h - 1, 0)
    d_hi = _POS_VALS[h] - av
    d_lo = av - _POS_VALS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_BITS[h] % 2 == 0))
    res = np.where(exact | pick_hi, _POS_BITS[h], _POS_BITS[lo])
    out[ok] = res
    out = out | np.where(np.signbit(p), 0x8000, 0).astype(np.uint32)
    return out.astype(np.uint16)


def nearest_bf16_bits_fraction(v: Fraction) -> int:
    """Same rounding for an exact rational (used on exact dot products)."""
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    if a == 0:
        return 0
    approx = float(a)
    h = int(np.searchsorted(_POS_VALS, approx, side="left"))
    # widen the bracket so the float conversion of ``a`` cannot mislead us
    lo_i = max(h - 2, 0)
    hi_i = min(h + 2, len(_POS_VALS) - 1)
    best = None
    for i in range(lo_i, hi_i + 1):
        d = abs(Fraction(float(_POS_VALS[i])) - a)
        key = (d, int(_POS_BITS[i]) % 2)
        if best is None or key < best[0]:
            best = (key, int(_POS_BITS[i]))
    return sign | best[1]
