"""Storage formats of the K/V pool -- TEST INFRASTRUCTURE ONLY (see the
package docstring for who may use it).

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
