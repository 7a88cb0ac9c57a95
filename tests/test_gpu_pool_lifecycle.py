"""Pool teardown returns every device buffer the pool made.

A pool allocates its working buffers on first use -- descriptors, partials,
host-call staging, the rotated queries of RoPE calls and the tensor-core
operand images -- and pkv_pool_free releases all of them.  Repeated
create / prefill with RoPE / free cycles must therefore not lose device
memory: a leaked image buffer here would be ~64 MB per cycle.
"""
from __future__ import annotations

import math

import pytest
import torch

import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool


def _cycle(H=32, KV=8, hd=128, bs=16, past=4000, n=64):
    kv_dim, q_dim = KV * hd, H * hd
    pool = GpuPool(-(-(past + n) // bs) + 4, 1, kv_dim, bs, max_seqs=2, max_blocks=-(-(past + n) // bs) + 2)
    try:
        s = pool.new_seq(past + n)
        pool.grow(s, past)
        pool.write_history(s, 0, torch.randn(past, kv_dim), torch.randn(past, kv_dim))
        Q = torch.randn(n, q_dim, device="cuda")
        K = torch.randn(n, kv_dim, device="cuda")
        V = torch.randn(n, kv_dim, device="cuda")
        out = torch.empty(n, q_dim, device="cuda")
        pkv.check(pkv.pkv_ensure_append(s, n))
        pkv.check(pkv.pkv_attn_batch_rope([s], [n], Q, K, V, H, KV, hd, 0, 1, 1.0 / math.sqrt(hd), 10000.0, out))
        pool.check_no_device_error()
        assert pkv.pkv_pool_last_work(pool.p)["prefill_tiles"] > 0
    finally:
        pool.close()
        del pool
    torch.cuda.synchronize()


@pytest.mark.gpu
def test_pool_free_releases_working_buffers():
    _cycle()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(4):
        _cycle()
    free1 = torch.cuda.mem_get_info()[0]
    assert free0 - free1 < 16 << 20, "device memory lost over 4 pool cycles: %d MB" % ((free0 - free1) >> 20)
