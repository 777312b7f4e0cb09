"""bf16 <-> float64 conversions for the oracle (test infrastructure only).

bf16 is the upper half of an IEEE binary32: 1 sign bit, 8 exponent bits, 7
stored mantissa bits.  Reading one is exact in float64.  Rounding a float64 to
bf16 uses round-to-nearest, ties-to-even on the 8 significant bits, done in
one step from float64 (no intermediate float32 rounding).
"""

from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16 / int16 array) as float64."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), as float64.

    For a finite nonzero x write x = m * 2**e with 0.5 <= |m| < 1 (frexp); bf16
    keeps 8 significant bits, so the result is rint(m * 2**8) * 2**(e - 8)
    with numpy's rint rounding halfway cases to even.  Zero stays zero.  The
    inputs of this oracle stay inside bf16's normal range (asserted).
    """
    x = np.asarray(x, dtype=np.float64)
    assert np.all(np.isfinite(x)), "round_to_bf16: non-finite input"
    m, e = np.frexp(x)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    nz = r != 0
    assert np.all(np.abs(r[nz]) >= 2.0 ** -126), "round_to_bf16: below bf16 normal range"
    assert np.all(np.abs(r) < 2.0 ** 128), "round_to_bf16: overflow"
    return r


def f64_to_bf16_bits(x) -> np.ndarray:
    """Bit patterns (uint16) of round_to_bf16(x)."""
    r = round_to_bf16(x).astype(np.float32)  # exact: r has 8 significant bits
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
