"""Storage formats of the K/V pool -- TEST INFRASTRUCTURE ONLY (see the
package docstring for who may use it).

Also the fp8 pool (another addition, no counterpart on the pages): a row is
stored as e4m3 of x / scale (scale a power of two), rounded to nearest with
ties to even and saturated to +-448, and read back as the e4m3 value times
scale.

The pages store K/V rows as f32 ("nx_f32_attn_paged.nx source": the pool
holds the rows the append writes).  A bf16 pool is an addition of this
library (no counterpart on the pages): every row is rounded once, when it is
written, to the nearest bfloat16 (ties to even), and attention reads the
rounded values back exactly.  bfloat16 keeps the sign, the 8 exponent bits and
the top 7 mantissa bits of an IEEE-754 binary32, so rounding to it is rounding
the binary32 bit pattern to its upper 16 bits.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x) -> np.ndarray:
    """Round float32 values to the nearest bfloat16, ties to even; returns
    float32 arrays holding the rounded values.  Finite inputs only."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = a.view(np.uint32).astype(np.uint64)
    upper = bits >> 16
    rest = bits & 0xFFFF
    # round up when the dropped half is above the midpoint, or at the midpoint
    # with an odd kept part
    up = (rest > 0x8000) | ((rest == 0x8000) & ((upper & 1) == 1))
    out = ((upper + up.astype(np.uint64)) << 16).astype(np.uint32)
    return out.view(np.float32).reshape(a.shape)


E4M3_MAX = 448.0


def round_e4m3(x, scale: float = 1.0) -> np.ndarray:
    """The value an fp8 pool reads back for float32 x: e4m3(x / scale) * scale,
    with e4m3 = 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, normal
    numbers from 2^-6, subnormals m * 2^-9, no infinities, largest finite
    448; rounding to nearest, ties to even, then saturation to +-448.
    `scale` must be a power of two.  Finite inputs only; returns float32."""
    m, e = np.frexp(float(scale))
    if m != 0.5:
        raise ValueError("scale must be a power of two")
    a = np.asarray(x, dtype=np.float64) / float(scale)     # exact: power of two
    mag = np.abs(a)
    with np.errstate(divide="ignore"):
        ex = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    ex = np.maximum(ex, -6.0)                                # subnormals share 2^-6's spacing
    ulp = np.exp2(ex - 3.0)                                  # 3 mantissa bits
    r = np.rint(mag / ulp) * ulp                             # nearest, ties to even
    r = np.minimum(r, E4M3_MAX)                              # satfinite
    return (np.sign(a) * r * float(scale)).astype(np.float32)
