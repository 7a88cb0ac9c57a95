"""The gate's deterministic small-integer input stream.

"nx_paged_kv_gate.nx source", the pg_lcg / pg_fill helpers and the "shared
deterministic inputs" block of main: the state advances as
``s = (s * 1103515245 + 12345) & 0x7fffffff`` (64-bit integer arithmetic, the
product stays below 2**62) BEFORE each use, and each value is the integer
``(s % 17) - 8`` in [-8, 8], stored as f32 (the "exact regime": every product
and short sum of such values is exact in f32).  One running state, seeded
20260709, fills Q1, K1, V1 (5 tokens), Q2, K2, V2 (1), Q3, K3, V3 (3), then
QA, KA, VA and QB, KB, VB (2 tokens each), in that order.
"""
from __future__ import annotations

import numpy as np

GATE_SEED = 20260709

# gate constants ("nx_paged_kv_gate.nx source", PG_* constants and main)
GATE_LAYERS = 2
GATE_HEADS = 4
GATE_KV_HEADS = 2
GATE_HEAD_DIM = 8
GATE_SCALE_BITS = 0x3E800000  # the f32 bit pattern of 0.25


def lcg_next(s: int) -> int:
    return (s * 1103515245 + 12345) & 0x7FFFFFFF


class LcgStream:
    def __init__(self, seed: int = GATE_SEED):
        self.state = seed

    def fill(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.float32)
        s = self.state
        for i in range(n):
            s = lcg_next(s)
            out[i] = (s % 17) - 8
        self.state = s
        return out


def gate_inputs(seed: int = GATE_SEED) -> dict:
    """All Q/K/V arrays of the gate, in the gate's fill order, shaped
    [tokens, dim] (q_dim = 32, kv_dim = 16)."""
    q_dim = GATE_HEADS * GATE_HEAD_DIM
    kv_dim = GATE_KV_HEADS * GATE_HEAD_DIM
    st = LcgStream(seed)
    out = {}
    for name, n in (("1", 5), ("2", 1), ("3", 3), ("A", 2), ("B", 2)):
        out["Q" + name] = st.fill(n * q_dim).reshape(n, q_dim)
        out["K" + name] = st.fill(n * kv_dim).reshape(n, kv_dim)
        out["V" + name] = st.fill(n * kv_dim).reshape(n, kv_dim)
    return out
