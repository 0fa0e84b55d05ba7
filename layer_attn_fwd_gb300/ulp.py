"""Units in the last place of the storage formats (measurement only).

ulp(x, fmt) is the spacing of the format's values in the binade of |x|:
2^(e - p) for 2^e <= |x| < 2^(e+1), p the stored fraction bits, and the fixed
subnormal spacing below the smallest normal binade.  Used to state the half
precision paths' errors in ULPs, the unit of the reduced-precision analysis
of "Shape-Aware Attention" (section Challenges we ran into: bf16's 7 fraction
bits make one ULP 2^(1-7) at magnitude 2.17).
"""
from __future__ import annotations

import numpy as np

# stored fraction bits, smallest normal exponent
FORMATS = {"bf16": (7, -126), "f16": (10, -14), "tf32": (10, -126), "f32": (23, -126)}


def ulp(x, fmt):
    """Spacing of `fmt` values at |x| (elementwise; x = 0 gives the subnormal spacing)."""
    p, emin = FORMATS[fmt]
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(a)              # a = m * 2^e with 0.5 <= m < 1, so floor(log2 a) = e - 1
    e = np.maximum(e - 1, emin)
    e = np.where(a > 0, e, emin)
    return np.ldexp(1.0, (e - p).astype(np.int64))


def unit_roundoff(fmt):
    """Largest relative error of round-to-nearest into `fmt` (normal range): 2^-(p+1)."""
    p, _ = FORMATS[fmt]
    return 2.0 ** -(p + 1)


def in_ulps(err, x, fmt):
    """An absolute error at value x, in ULPs of `fmt` there."""
    return np.asarray(err, dtype=np.float64) / ulp(x, fmt)
