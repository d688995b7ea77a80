"""bfloat16 <-> float64 for the oracle (test infrastructure only).

bf16 is the top half of an IEEE binary32: 1 sign bit, 8 exponent bits, 7
stored fraction bits.  Decoding is exact; encoding rounds to nearest, ties to
even, straight from float64 (one rounding).
"""

import numpy as np


def bf16_bits_to_f64(bits):
    """Exact value of bf16 bit patterns (uint16 array) as float64."""
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """Round float64 values to the nearest bf16 (ties to even); return uint16 bits.

    A finite x = m * 2**e with 0.5 <= |m| < 1 keeps 8 significant bits, so the
    spacing of bf16 numbers around x is 2**(e - 8); below the smallest normal
    (2**-126) the spacing stays 2**-133.  ``np.rint`` rounds half to even, and
    x / spacing is exact in float64, so the rounding is exact.  Values that
    round beyond the largest finite bf16 become infinities.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    xf = x[finite]
    _, e = np.frexp(xf)
    e = np.maximum(e, -125)
    spacing = np.ldexp(1.0, e - 8)
    r = np.rint(xf / spacing) * spacing
    largest = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > largest, np.copysign(np.inf, r), r)
    out[finite] = r
    out[~finite] = x[~finite]
    # every value is now a bf16 number, hence exact in float32: keep its top half
    return (out.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
