"""Seeded synthetic workloads: shapes, length mixes and tensor draws.

Nothing here computes attention or touches pool metadata; it only draws
numbers.  Every workload is seeded (20260709 + its index) so a test and the
benchmark see the same inputs.

Workloads (attention shape of Qwen3-4B where stated -- 32 query heads sharing 8
kv heads of width 128, from the header of "nx_f32_gqa_attention.nx source"):

* ``batched_decode_m64``      M=64 rows, n_q=1, past length uniform in
                              [512, 4096], block_size 16, 1 layer.
* ``chunked_prefill``         8 sequences, 2048 past tokens plus one 512-token
                              chunk, 4 layers, block_size 16.
* ``continuous_batching_m256`` M=256 rows, n_q=1, past length log-uniform in
                              [128, 32768] (exp of a uniform draw, rounded),
                              block_size 16, 1 layer, pool of 600 000 blocks.
* ``shared_prefix_forks``     one 8192-token prefix, 128 forks each appending
                              a 1..256-token divergent chunk, block_size 16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BASE_SEED = 20260709


@dataclass
class Workload:
    name: str
    n_heads: int
    n_kv_heads: int
    head_dim: int
    n_layers: int
    block_size: int
    n_blocks: int
    past_len: np.ndarray            # [M] tokens already in each sequence
    n_q: np.ndarray                 # [M] rows appended + attended this step
    seed: int
    extra: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        return int(self.past_len.shape[0])

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))

    def max_tokens(self) -> int:
        return int((self.past_len + self.n_q).max())


def _blocks_for(lengths, bs: int) -> int:
    return int(sum(-(-int(x) // bs) for x in lengths))


def batched_decode_m64(seed: int = BASE_SEED + 1) -> Workload:
    rng = np.random.default_rng(seed)
    past = rng.integers(512, 4096, size=64, endpoint=True).astype(np.int64)
    n_q = np.ones(64, dtype=np.int64)
    need = _blocks_for(past + n_q, 16)
    return Workload("batched_decode_m64", 32, 8, 128, 1, 16, int(need * 1.1) + 8,
                    past, n_q, seed)


def chunked_prefill(seed: int = BASE_SEED + 2) -> Workload:
    past = np.full(8, 2048, dtype=np.int64)
    n_q = np.full(8, 512, dtype=np.int64)
    need = _blocks_for(past + n_q, 16)
    return Workload("chunked_prefill", 32, 8, 128, 4, 16, int(need * 1.1) + 8,
                    past, n_q, seed)


def continuous_batching_m256(seed: int = BASE_SEED + 3, n_blocks: int = 600_000) -> Workload:
    rng = np.random.default_rng(seed)
    u = rng.uniform(math.log(128.0), math.log(32768.0), size=256)
    past = np.clip(np.rint(np.exp(u)), 128, 32768).astype(np.int64)
    n_q = np.ones(256, dtype=np.int64)
    return Workload("continuous_batching_m256", 32, 8, 128, 1, 16, n_blocks,
                    past, n_q, seed)


def continuous_batching_small(seed: int = BASE_SEED + 3) -> Workload:
    """A smaller draw of the continuous-batching mix for profiler captures:
    M=64, lengths log-uniform in [128, 8192], a 32 768-block pool (4.3 GB);
    each step still reads ~0.8 GB of K/V, well above the L2."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(math.log(128.0), math.log(8192.0), size=64)
    past = np.clip(np.rint(np.exp(u)), 128, 8192).astype(np.int64)
    return Workload("continuous_batching_small", 32, 8, 128, 1, 16, 32768, past,
                    np.ones(64, dtype=np.int64), seed)


def shared_prefix_forks(seed: int = BASE_SEED + 4, prefix: int = 8192,
                        n_forks: int = 128) -> Workload:
    rng = np.random.default_rng(seed)
    div = rng.integers(1, 256, size=n_forks, endpoint=True).astype(np.int64)
    w = Workload("shared_prefix_forks", 32, 8, 128, 1, 16, 4096,
                 np.full(n_forks, prefix, dtype=np.int64), div, seed)
    w.extra["prefix"] = prefix
    return w


def scaled(w: Workload, max_len: int) -> Workload:
    """A smaller copy of ``w`` for quick checks: lengths clipped to ``max_len``."""
    past = np.minimum(w.past_len, max_len)
    return Workload(w.name + "_clip%d" % max_len, w.n_heads, w.n_kv_heads, w.head_dim,
                    w.n_layers, w.block_size,
                    _blocks_for(past + w.n_q, w.block_size) + 64,
                    past, w.n_q.copy(), w.seed, dict(w.extra))


def release_order(n_blocks: int, seed: int) -> np.ndarray:
    """A seeded permutation of block ids.  Allocating every block and then
    releasing them in this order leaves the free list shuffled, so later
    allocations scatter each sequence over the pool."""
    return np.random.default_rng(seed ^ 0x5EED).permutation(n_blocks)


def normal(shape, seed: int, device="cpu"):
    """f32 N(0, 1) draws from a seeded torch generator on ``device``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)


def uniform_ints(shape, lo: int, hi: int, seed: int) -> np.ndarray:
    """Small integers in [lo, hi] as f32 (exact products and sums)."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi, size=shape, endpoint=True).astype(np.float32)
