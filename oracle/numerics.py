"""Float64 reference rounding to bfloat16.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
module.  It shares no code with the CUDA path.

bfloat16 is binary32 with the fraction cut to 7 bits: a sign, the same 8-bit exponent
(bias 127, normal numbers from 2^-126, subnormals spaced 2^-133) and 8 significant bits
for normal numbers.  Rounding a real number to it takes the nearest representable value
and, on a tie, the one whose last significand bit is 0 (round to nearest, ties to even);
magnitudes at or past the midpoint between the largest finite value (2^128 - 2^120) and
2^128 round to infinity.

Pins (tests/test_oracle_numerics.py): torch's float32 -> bfloat16 conversion on values
exactly representable in float32 across the whole exponent range (subnormals included),
and hand-worked ties.
"""
from __future__ import annotations

import numpy as np

__all__ = ["to_bf16"]

_MAX_FINITE = 2.0 ** 128 - 2.0 ** 120
_OVERFLOW = 2.0 ** 128 - 2.0 ** 119      # the midpoint to the next power: ties go to infinity


def to_bf16(x):
    """Nearest bfloat16 value (ties to even) of every float64 value of x, as float64."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    a = np.abs(x)
    # normal range: x = m 2^e with 0.5 <= |m| < 1, so 8 significant bits are m * 2^8
    m, e = np.frexp(x)
    normal = a >= 2.0 ** -126
    out[normal] = np.ldexp(np.rint(np.ldexp(m[normal], 8)), e[normal] - 8)
    # subnormal range: a fixed spacing of 2^-133
    sub = ~normal
    out[sub] = np.ldexp(np.rint(np.ldexp(x[sub], 133)), -133)
    over = a >= _OVERFLOW
    out[over] = np.copysign(np.inf, x[over])
    special = ~np.isfinite(x)
    out[special] = x[special]
    return out
