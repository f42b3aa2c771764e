"""bf16 conversions on raw bit patterns -- oracle side (test infrastructure).

The dense bf16 workload widens bf16 inputs to fp32 exactly, accumulates in
fp32 and rounds once to bf16 at the output.  bf16 is the top 16 bits of an
IEEE binary32, so:

* widening: place the 16 bits above 16 zero bits;
* narrowing: round-to-nearest, ties-to-even, on the 16 bits that are dropped.
  Adding 0x7FFF plus the lowest kept bit and truncating does exactly that (a
  carry out of the mantissa bumps the exponent; the largest finite values
  round to infinity, as IEEE 754 requires).  NaNs keep their sign and top
  payload bits and are made quiet.
"""

import numpy as np


def widen(bits):
    """bf16 bit patterns (uint16) -> float32, exactly."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_rne(x):
    """float32 values -> bf16 bit patterns (uint16), round-to-nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint32)
    is_nan = np.isnan(x)
    if is_nan.any():
        quiet = ((u >> np.uint64(16)).astype(np.uint32)) | np.uint32(0x0040)
        rounded = np.where(is_nan, quiet, rounded)
    return rounded.astype(np.uint16)
