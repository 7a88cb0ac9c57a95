"""Contiguous K/V history of one sequence -- TEST INFRASTRUCTURE ONLY (oracle).

The pages gate the paged path against a contiguous-cache twin ("nx_paged_kv_gate.nx
source", EQUIV and FORK sections: nx_f32_kv_cache_alloc(n_layers, n_kv_heads,
max_seq, head_dim), nx_f32_attn_with_cache, nx_f32_kv_cache_advance).  This class
is that twin, written from its call sites: per layer a stripe of ``max_seq`` rows
of ``n_kv_heads * head_dim`` floats; a call appends ``n_tokens`` rows at
``seq_len`` and attends over ``total_k = seq_len + n_tokens``; the length moves
only on ``advance`` (caller contract, "nx_f32_attn_paged.nx source" header).

Truncation (the REWIND section of the gate) only moves ``seq_len`` back: rows
past it are overwritten by the next append before anything reads them.
"""
from __future__ import annotations

import copy

import numpy as np

from . import attend, OK, ERR_BAD_DIM, ERR_BAD_GQA

ERR_SEQ = 3


class ContiguousCache:
    def __init__(self, n_layers: int, n_kv_heads: int, max_seq: int, head_dim: int):
        self.n_layers = n_layers
        self.n_kv_heads = n_kv_heads
        self.max_seq = max_seq
        self.head_dim = head_dim
        self.kv_dim = n_kv_heads * head_dim
        self.K = np.zeros((n_layers, max_seq, self.kv_dim), dtype=np.float32)
        self.V = np.zeros((n_layers, max_seq, self.kv_dim), dtype=np.float32)
        self.seq_len = 0

    def attn_with_cache(self, Q, K_new, V_new, n_tokens: int, n_heads: int,
                        n_kv_heads: int, head_dim: int, layer: int, causal: int,
                        scale: float):
        """Append this layer's rows, then attend (same checks and order as
        nx_f32_attn_with_paged, "nx_f32_attn_paged.nx source": sizes -> 1,
        grouping -> 2, storage -> 3).  Returns ``(rc, out)``."""
        if n_tokens <= 0 or n_heads <= 0 or n_kv_heads <= 0 or head_dim <= 0:
            return ERR_BAD_DIM, None
        if n_heads % n_kv_heads != 0:
            return ERR_BAD_GQA, None
        if (n_kv_heads != self.n_kv_heads or head_dim != self.head_dim
                or not 0 <= layer < self.n_layers
                or self.seq_len + n_tokens > self.max_seq):
            return ERR_SEQ, None
        kn = np.asarray(K_new, dtype=np.float32).reshape(n_tokens, self.kv_dim)
        vn = np.asarray(V_new, dtype=np.float32).reshape(n_tokens, self.kv_dim)
        s = self.seq_len
        self.K[layer, s:s + n_tokens] = kn
        self.V[layer, s:s + n_tokens] = vn
        total_k = s + n_tokens
        rc, out = attend(Q, self.K[layer, :total_k], self.V[layer, :total_k], n_tokens,
                         total_k, n_heads, n_kv_heads, head_dim, causal, scale)
        return rc, out

    def advance(self, n: int) -> None:
        self.seq_len += n

    def truncate(self, new_len: int) -> None:
        if not 0 <= new_len <= self.seq_len:
            raise ValueError("truncate outside [0, seq_len]")
        self.seq_len = new_len

    def fork(self) -> "ContiguousCache":
        return copy.deepcopy(self)

    def history(self, layer: int):
        """The visible K and V rows of ``layer``: [seq_len, kv_dim] each."""
        return self.K[layer, :self.seq_len], self.V[layer, :self.seq_len]


__all__ = ["ContiguousCache", "OK"]
