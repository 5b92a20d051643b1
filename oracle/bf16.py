"""bf16 storage helpers for the oracle (test infrastructure only).

bfloat16 values are carried as their raw 16-bit patterns in ``numpy.uint16`` arrays:
numpy has no bf16 type.  A bf16 pattern is the upper half of the fp32 pattern with the
same sign, exponent and leading 7 mantissa bits, so widening is exact.

Rounding fp64 -> bf16 is done in one step, round-to-nearest-even on 8 significant bits,
without going through fp32 first (that would round twice).
"""

import numpy as np


def bf16_bits_to_f64(bits):
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """Round float64 values to bf16, nearest-even, and return the uint16 patterns.

    For a finite x = m * 2**e with 0.5 <= |m| < 1, bf16 keeps 8 significant bits, so the
    rounding quantum is 2**(e-8); below the smallest normal (2**-126) the quantum stays at
    the subnormal step 2**-133.  ``np.rint`` rounds half to even.  Values that round past
    the largest finite bf16 become +-inf; NaN stays NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)
        q = np.maximum(e - 8, -133)
        r = np.ldexp(np.rint(np.ldexp(x, -q)), q)
        f32 = r.astype(np.float32)
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits
