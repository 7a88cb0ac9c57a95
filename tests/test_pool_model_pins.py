"""Pins for the pool / page-table / refcount model (CPU only).

The model is tied to the gate's own known answers ("nx_paged_kv_gate.nx
source": KAT ids 0,1,2,-1 and recycling; refcount 2 on a shared prompt block
after a fork; divergence with refcount 1 after both forks append; truncate
releasing blocks) and to invariants that any correct refcounted pool keeps:
every block is free exactly when its refcount is 0, and its refcount equals
the number of page-table entries (plus caller-held ids) that name it.
"""
import json
import os
import random

import pytest

from oracle.pool_model import (PoolModel, OK, ERR_ARG, ERR_CAPACITY, ERR_EXHAUSTED, ERR_SEQ)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kat_golden():
    g = json.load(open(os.path.join(GOLDEN, "pool_kat.json")))
    p = PoolModel(g["n_blocks"], 2, 16, 4, 4, 16)
    assert [p.alloc_block() for _ in g["allocs"]] == g["allocs"]
    assert p.unref_block(g["release"]) == OK
    assert p.alloc_block() == g["realloc"]
    p.check_invariants(extra_refs=[0, 1, 2])


def _prefill(p, s, n):
    assert p.ensure_append(s, n) == OK
    assert p.can_append(s, n) == OK
    assert p.advance(s, n) == OK


def test_fork_literal_gate_checks_bs8():
    """At block_size 8 the 5-token prompt sits in one partial block, so the
    gate's literal checks on pt[0] apply verbatim."""
    p = PoolModel(16, 2, 16, 8, 8, 8)
    a = p.seq_new(64)
    _prefill(p, a, 5)
    b = p.seq_fork(a)
    assert p.refcnt[a.pt[0]] == 2 and a.pt == b.pt
    _prefill(p, a, 2)          # a writes into the shared block: copy-on-append
    _prefill(p, b, 2)          # b is now the block's only holder: no copy
    assert a.pt[0] != b.pt[0]
    assert p.refcnt[a.pt[0]] == 1 and p.refcnt[b.pt[0]] == 1
    p.check_invariants()


def test_fork_tail_only_cow_bs4():
    """At block_size 4 the prompt fills block 0 and starts block 1; only the
    written tail block diverges, the full prefix block stays shared."""
    p = PoolModel(16, 2, 16, 4, 8, 16)
    a = p.seq_new(64)
    _prefill(p, a, 5)
    b = p.seq_fork(a)
    assert p.refcnt[a.pt[0]] == 2 and p.refcnt[a.pt[1]] == 2
    _prefill(p, a, 2)
    _prefill(p, b, 2)
    assert a.pt[0] == b.pt[0] and p.refcnt[a.pt[0]] == 2
    assert a.pt[1] != b.pt[1]
    assert p.refcnt[a.pt[1]] == 1 and p.refcnt[b.pt[1]] == 1
    p.check_invariants()


def test_append_into_shared_block_is_refused():
    p = PoolModel(16, 1, 16, 4, 8, 16)
    a = p.seq_new(64)
    _prefill(p, a, 5)
    b = p.seq_fork(a)
    assert p.can_append(a, 1) == ERR_SEQ      # block 1 is shared and unensured
    assert p.ensure_append(a, 1) == OK
    assert p.can_append(a, 1) == OK
    assert p.can_append(b, 1) == OK           # b now holds block 1 alone
    p.check_invariants()


def test_truncate_releases_tail_blocks():
    p = PoolModel(16, 1, 16, 4, 8, 16)
    a = p.seq_new(64)
    _prefill(p, a, 10)                         # blocks for positions 0..11
    assert len(a.pt) == 3
    tail = list(a.pt[2:])
    assert p.seq_truncate(a, 5) == OK          # keep ceil(5/4) = 2 blocks
    assert len(a.pt) == 2 and a.len == 5
    assert all(p.refcnt[b] == 0 for b in tail)
    assert p.seq_truncate(a, 6) == ERR_ARG     # cannot grow by truncation
    assert p.seq_truncate(a, -1) == ERR_ARG
    p.check_invariants()


def test_truncate_then_reappend_reuses_same_blocks():
    """Released last-first onto a LIFO stack, the blocks come back in the
    same order when the sequence grows again."""
    p = PoolModel(32, 1, 16, 4, 8, 16)
    a = p.seq_new(64)
    _prefill(p, a, 16)
    before = list(a.pt)
    assert p.seq_truncate(a, 4) == OK
    _prefill(p, a, 12)
    assert a.pt == before


def test_exhaustion_is_all_or_nothing():
    p = PoolModel(4, 1, 16, 4, 8, 16)
    a = p.seq_new(64)
    b = p.seq_new(64)
    _prefill(p, a, 8)                          # 2 blocks used, 2 free
    snap = (list(p.free), list(p.refcnt), list(a.pt), list(b.pt))
    assert p.ensure_append_batch([a, b], [4, 8]) == ERR_EXHAUSTED   # needs 1 + 2
    assert (list(p.free), list(p.refcnt), list(a.pt), list(b.pt)) == snap
    assert p.ensure_append_batch([a, b], [4, 4]) == OK
    assert p.ensure_append(b, 9) == ERR_EXHAUSTED
    p.check_invariants()


def test_capacity_and_argument_errors():
    p = PoolModel(16, 1, 16, 4, 8, 4)
    assert p.seq_new(17) is None               # 5 blocks > max_blocks_per_seq
    a = p.seq_new(6)
    assert p.ensure_append(a, 7) == ERR_CAPACITY
    assert p.ensure_append(a, 0) == ERR_ARG
    assert p.ensure_append_batch([a, a], [1, 1]) == ERR_ARG
    assert p.advance(a, 1) == ERR_SEQ          # no block covers position 0 yet
    assert p.unref_block(3) == ERR_ARG         # not allocated
    assert p.unref_block(99) == ERR_ARG


def test_fresh_pops_ascend_and_shuffle_through_api():
    p = PoolModel(10, 1, 16, 4, 4, 8)
    ids = [p.alloc_block() for _ in range(10)]
    assert ids == list(range(10))
    order = [3, 7, 1, 9, 0, 2, 8, 4, 6, 5]
    for b in order:
        p.unref_block(b)
    assert [p.alloc_block() for _ in range(10)] == order[::-1]


def test_cow_in_batch_counts_shared_blocks_once():
    """Two forks sharing a tail block in one batch: the first copies, the
    second is then the sole holder and writes in place."""
    p = PoolModel(8, 1, 16, 4, 8, 8)
    a = p.seq_new(32)
    _prefill(p, a, 5)
    b = p.seq_fork(a)
    free_before = len(p.free)
    assert p.ensure_append_batch([a, b], [1, 1]) == OK
    assert len(p.free) == free_before - 1
    assert a.pt[1] != b.pt[1]
    p.check_invariants()


@pytest.mark.parametrize("seed", range(8))
def test_random_ops_keep_invariants(seed):
    rng = random.Random(seed)
    p = PoolModel(48, 2, 16, rng.choice([1, 2, 4, 8]), 12, 64)
    held = []
    for _ in range(600):
        op = rng.randrange(9)
        seqs = list(p.seqs)
        if op == 0 and len(seqs) < 10:
            p.seq_new(rng.randrange(1, 60))
        elif op == 1 and seqs:
            p.seq_fork(rng.choice(seqs))
        elif op == 2 and seqs:
            p.seq_free(rng.choice(seqs))
        elif op == 3 and seqs:
            s = rng.choice(seqs)
            p.seq_truncate(s, rng.randrange(0, s.len + 2))
        elif op in (4, 5) and seqs:
            k = rng.randrange(1, min(4, len(seqs)) + 1)
            batch = rng.sample(seqs, k)
            ns = [rng.randrange(1, 9) for _ in batch]
            if p.ensure_append_batch(batch, ns) == OK:
                for s, n in zip(batch, ns):
                    assert p.can_append(s, n) == OK
                    assert p.advance(s, n) == OK
        elif op == 6:
            b = p.alloc_block()
            if b >= 0:
                held.append(b)
        elif op == 7 and held:
            p.unref_block(held.pop(rng.randrange(len(held))))
        p.check_invariants(extra_refs=held)
