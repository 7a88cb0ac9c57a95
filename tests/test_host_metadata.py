"""Pool, page-table and refcount state of the C++ host core, bit-exact against
the oracle's pool model (CPU only: host-only pools make no CUDA call).

Random operation sequences (seq_new, fork, free, truncate, batched
ensure_append / advance, alloc_block / unref_block) are applied to both; after
every operation the return codes, every block's refcount, every live page
table, every length and the free-block count must agree, and block ids handed
out by alloc must be the same ids.
"""
import json
import os
import random

import pytest

import paged_kv_gqa_nx_gb300 as pkv
from oracle.pool_model import PoolModel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def host_pool(n_blocks, n_layers, kv_dim, bs, max_seqs, max_blocks):
    p = pkv.pkv_pool_new(n_blocks, n_layers, kv_dim, bs, None, None, max_seqs, max_blocks, None,
                         pkv.PKV_POOL_HOST_ONLY)
    assert p, pkv.pkv_last_error()
    return p


def test_kat_through_c_abi():
    g = json.load(open(os.path.join(GOLDEN, "pool_kat.json")))
    p = host_pool(g["n_blocks"], 2, 16, 4, 4, 16)
    try:
        assert [pkv.pkv_alloc_block(p) for _ in g["allocs"]] == g["allocs"]
        assert pkv.pkv_unref_block(p, g["release"]) == pkv.PKV_OK
        assert pkv.pkv_alloc_block(p) == g["realloc"]
        assert pkv.pkv_unref_block(p, 7) == pkv.PKV_ERR_ARG
    finally:
        pkv.pkv_pool_free(p)


def test_gate_fork_refcounts_through_c_abi():
    """FORK section of the gate at block_size 8 (the literal checks) and 4
    (tail-only copy-on-append)."""
    for bs in (8, 4):
        p = host_pool(16, 2, 16, bs, 8, 16)
        try:
            a = pkv.pkv_seq_new(p, 64)
            assert pkv.pkv_ensure_append(a, 5) == 0 and pkv.pkv_advance(a, 5) == 0
            b = pkv.pkv_seq_fork(a)
            pa = pkv.pkv_seq_page_table(a)
            assert pkv.pkv_refcnt(p, pa[0]) == 2
            for s in (a, b):
                assert pkv.pkv_ensure_append(s, 2) == 0 and pkv.pkv_advance(s, 2) == 0
            pa, pb = pkv.pkv_seq_page_table(a), pkv.pkv_seq_page_table(b)
            tail = 4 // bs
            assert pa[tail] != pb[tail]
            assert pkv.pkv_refcnt(p, pa[tail]) == 1 and pkv.pkv_refcnt(p, pb[tail]) == 1
            if bs == 4:
                assert pa[0] == pb[0] and pkv.pkv_refcnt(p, pa[0]) == 2
            assert pkv.pkv_seq_truncate(a, 5) == 0
            assert pkv.pkv_seq_len(a) == 5
        finally:
            pkv.pkv_pool_free(p)


class Twin:
    """The C pool and the model pool driven in lockstep."""

    def __init__(self, n_blocks, n_layers, kv_dim, bs, max_seqs, max_blocks):
        self.c = host_pool(n_blocks, n_layers, kv_dim, bs, max_seqs, max_blocks)
        self.m = PoolModel(n_blocks, n_layers, kv_dim, bs, max_seqs, max_blocks)
        self.pairs = []   # (c handle, model seq)
        self.held = []    # ids from alloc_block

    def compare(self):
        m, c = self.m, self.c
        assert pkv.pkv_pool_free_blocks(c) == len(m.free)
        for b in range(m.n_blocks):
            assert pkv.pkv_refcnt(c, b) == m.refcnt[b], b
        for hc, sm in self.pairs:
            assert pkv.pkv_seq_page_table(hc) == sm.pt
            assert pkv.pkv_seq_len(hc) == sm.len
            assert pkv.pkv_seq_slot(hc) == sm.slot
        m.check_invariants(extra_refs=self.held)

    def close(self):
        pkv.pkv_pool_free(self.c)


@pytest.mark.parametrize("seed", range(12))
def test_random_ops_bit_exact_vs_model(seed):
    rng = random.Random(1000 + seed)
    bs = rng.choice([1, 2, 3, 4, 8, 16])
    t = Twin(rng.choice([24, 48, 96]), 2, 16, bs, 10, 64 // bs + 8)
    try:
        for _ in range(500):
            op = rng.randrange(10)
            if op == 0 and len(t.pairs) < 9:
                mt = rng.randrange(-1, 70)
                hc = pkv.pkv_seq_new(t.c, mt)
                sm = t.m.seq_new(mt)
                assert (hc is None) == (sm is None)
                if hc:
                    t.pairs.append((hc, sm))
            elif op == 1 and t.pairs:
                hc, sm = rng.choice(t.pairs)
                hc2, sm2 = pkv.pkv_seq_fork(hc), t.m.seq_fork(sm)
                assert (hc2 is None) == (sm2 is None)
                if hc2:
                    t.pairs.append((hc2, sm2))
            elif op == 2 and t.pairs:
                i = rng.randrange(len(t.pairs))
                hc, sm = t.pairs.pop(i)
                assert pkv.pkv_seq_free(hc) == t.m.seq_free(sm)
            elif op == 3 and t.pairs:
                hc, sm = rng.choice(t.pairs)
                nl = rng.randrange(-1, sm.len + 2)
                assert pkv.pkv_seq_truncate(hc, nl) == t.m.seq_truncate(sm, nl)
            elif op in (4, 5, 6) and t.pairs:
                k = rng.randrange(1, min(4, len(t.pairs)) + 1)
                batch = rng.sample(t.pairs, k)
                if rng.random() < 0.05:
                    batch = batch + [batch[0]]          # duplicate -> argument error
                ns = [rng.choice([1, 1, 2, 3, 5, 9, 17, 0, -1]) for _ in batch]
                rc_c = pkv.pkv_ensure_append_batch([b[0] for b in batch], ns)
                rc_m = t.m.ensure_append_batch([b[1] for b in batch], ns)
                assert rc_c == rc_m
                if rc_m == 0 and rng.random() < 0.9:
                    rc_c = pkv.pkv_advance_batch([b[0] for b in batch], ns)
                    rc_m = t.m.advance_batch([b[1] for b in batch], ns)
                    assert rc_c == rc_m == 0
            elif op == 7 and t.pairs and rng.random() < 0.3:
                k = rng.randrange(1, min(4, len(t.pairs)) + 1)
                batch = rng.sample(t.pairs, k)
                nls = [rng.randrange(-1, b[1].len + 2) for b in batch]
                assert pkv.pkv_seq_truncate_batch([b[0] for b in batch], nls) == \
                    t.m.seq_truncate_batch([b[1] for b in batch], nls)
            elif op == 7 and t.pairs:
                hc, sm = rng.choice(t.pairs)
                n = rng.randrange(-1, 6)
                assert pkv.pkv_advance(hc, n) == t.m.advance(sm, n)
            elif op == 8:
                bc, bm = pkv.pkv_alloc_block(t.c), t.m.alloc_block()
                assert bc == bm
                if bm >= 0:
                    t.held.append(bm)
            elif op == 9 and t.held:
                b = t.held.pop(rng.randrange(len(t.held)))
                assert pkv.pkv_unref_block(t.c, b) == t.m.unref_block(b)
            t.compare()
    finally:
        t.close()


def test_shuffled_pool_through_api():
    """Allocating every block and releasing them in a seeded order makes later
    allocations follow the reverse of that order (LIFO)."""
    import numpy as np
    from synth.workloads import release_order
    n = 64
    t = Twin(n, 1, 16, 16, 4, 8)
    try:
        ids = [pkv.pkv_alloc_block(t.c) for _ in range(n)]
        [t.m.alloc_block() for _ in range(n)]
        assert ids == list(range(n))
        order = release_order(n, 7)
        for b in order:
            assert pkv.pkv_unref_block(t.c, int(b)) == t.m.unref_block(int(b)) == 0
        got = [pkv.pkv_alloc_block(t.c) for _ in range(n)]
        assert got == [int(b) for b in order[::-1]] == [t.m.alloc_block() for _ in range(n)]
    finally:
        t.close()


def test_capacity_errors_match():
    t = Twin(8, 1, 16, 4, 2, 4)
    try:
        assert pkv.pkv_seq_new(t.c, 17) is None and t.m.seq_new(17) is None
        a, am = pkv.pkv_seq_new(t.c, 6), t.m.seq_new(6)
        b, bm = pkv.pkv_seq_new(t.c, 6), t.m.seq_new(6)
        assert pkv.pkv_seq_new(t.c, 6) is None and t.m.seq_new(6) is None   # max_seqs live
        t.pairs = [(a, am), (b, bm)]
        assert pkv.pkv_ensure_append(a, 7) == t.m.ensure_append(am, 7) == pkv.PKV_ERR_CAPACITY
        assert pkv.pkv_seq_fork(a) is None and t.m.seq_fork(am) is None
        t.compare()
    finally:
        t.close()


def test_image_cache_needs_a_device_pool():
    # the operand-image cache lives in device memory: a host-only pool, a NULL
    # pool and a negative size are argument errors, and nothing is allocated
    p = host_pool(8, 1, 16, 4, 2, 4)
    try:
        assert pkv.pkv_pool_set_image_cache(p, 1 << 20) == pkv.PKV_ERR_ARG
        assert pkv.pkv_pool_set_image_cache(p, 0) == pkv.PKV_ERR_ARG
        assert pkv.pkv_pool_set_image_cache(None, 1 << 20) == pkv.PKV_ERR_ARG
        assert "device pool" in pkv.pkv_last_error()
        assert pkv.pkv_alloc_block(p) == 0   # the pool itself is untouched
    finally:
        pkv.pkv_pool_free(p)
