"""Paged KV pool metadata model -- TEST INFRASTRUCTURE ONLY (oracle).

A plain model of the refcounted block pool and the per-sequence page tables,
written from the pages' call sites (the pool module itself is imported by the
pages but never listed):

* "nx_paged_kv_gate.nx source", KAT section: a pool of 3 blocks hands out ids
  0, 1, 2, then -1 on exhaustion; a freed id is handed out again.
* same page, FORK section: a fork shares its parent's blocks (refcount 2);
  after both forks append, each owns a private copy of the block it wrote
  (refcount 1) -- copy-on-append.
* same page, REWIND section: truncate releases the blocks past the new length
  ("truncate unref" in the header) and a later append overwrites the rest.
* "nx_f32_attn_paged.nx source", caller contract: ensure_append once per step
  before layer 0, append + attend per layer, advance once after all layers.
* "nx_f32_llama_v4b.nx source", Stack section: ensure_append(seq_r, 1) for
  every sequence before the layers, advance(seq_r, 1) for every one after.

Readings where the pages are silent (each is also listed in the design notes):

1. Free list: a LIFO stack whose fresh pops ascend 0, 1, 2, ...
2. Copy-on-append privatises only the blocks the append will write into
   (indices floor(len/bs) .. floor((len+n-1)/bs)) that are shared
   (refcount > 1): a new block is taken, the old one is unreferenced.
   Within one call the copies come first, in ascending index order, then the
   new tail blocks in ascending index order.
3. ensure_append is all-or-nothing: on exhaustion or when len + n exceeds the
   sequence's max_tokens nothing changes.  The batch form is all-or-nothing
   over the whole batch (simulated on a copy, then committed).
4. truncate(new_len) needs 0 <= new_len <= len and releases the blocks with
   index >= ceil(new_len/bs), last block first; seq_free releases all blocks,
   last first.
5. seq_new(pool, max_tokens): max_tokens is the capacity; the page table holds
   ceil(max_tokens/bs) entries at most.
6. Appending n rows needs the blocks covering [len, len+n) to exist and to be
   private (refcount 1); otherwise the append fails with the storage error.
7. Duplicate sequences inside one batch call are an argument error.

Status codes match the library's: 0 ok, 1 bad dim, 2 bad GQA, 3 sequence /
storage error, 4 pool exhausted, 5 capacity, 6 bad argument.
"""
from __future__ import annotations

import copy

OK = 0
ERR_BAD_DIM = 1
ERR_BAD_GQA = 2
ERR_SEQ = 3
ERR_EXHAUSTED = 4
ERR_CAPACITY = 5
ERR_ARG = 6


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


class SeqModel:
    def __init__(self, slot: int, max_tokens: int):
        self.slot = slot
        self.max_tokens = max_tokens
        self.len = 0
        self.pt: list[int] = []
        self.alive = True


class PoolModel:
    def __init__(self, n_blocks: int, n_layers: int, kv_dim: int, block_size: int,
                 max_seqs: int, max_blocks_per_seq: int):
        if min(n_blocks, n_layers, kv_dim, block_size, max_seqs, max_blocks_per_seq) <= 0:
            raise ValueError("pool sizes must be positive")
        self.n_blocks = n_blocks
        self.n_layers = n_layers
        self.kv_dim = kv_dim
        self.bs = block_size
        self.max_seqs = max_seqs
        self.max_blocks_per_seq = max_blocks_per_seq
        # stack top is the list's end: the first pops give 0, 1, 2, ...
        self.free = list(range(n_blocks - 1, -1, -1))
        self.refcnt = [0] * n_blocks
        self.free_slots = list(range(max_seqs - 1, -1, -1))
        self.seqs: list[SeqModel] = []

    # ---- blocks (KAT section) -------------------------------------------------
    def alloc_block(self) -> int:
        if not self.free:
            return -1
        b = self.free.pop()
        self.refcnt[b] = 1
        return b

    def unref_block(self, b: int) -> int:
        if not 0 <= b < self.n_blocks or self.refcnt[b] <= 0:
            return ERR_ARG
        self.refcnt[b] -= 1
        if self.refcnt[b] == 0:
            self.free.append(b)
        return OK

    # ---- sequences --------------------------------------------------------------
    def seq_new(self, max_tokens: int):
        if max_tokens <= 0 or _ceil_div(max_tokens, self.bs) > self.max_blocks_per_seq:
            return None
        if not self.free_slots:
            return None
        s = SeqModel(self.free_slots.pop(), max_tokens)
        self.seqs.append(s)
        return s

    def seq_fork(self, parent: SeqModel):
        if parent is None or not parent.alive or not self.free_slots:
            return None
        child = SeqModel(self.free_slots.pop(), parent.max_tokens)
        child.len = parent.len
        child.pt = list(parent.pt)
        for b in child.pt:
            self.refcnt[b] += 1
        self.seqs.append(child)
        return child

    def seq_free(self, s: SeqModel) -> int:
        if s is None or not s.alive:
            return ERR_ARG
        for b in reversed(s.pt):
            self.unref_block(b)
        s.pt = []
        s.alive = False
        self.free_slots.append(s.slot)
        self.seqs.remove(s)
        return OK

    def seq_truncate(self, s: SeqModel, new_len: int) -> int:
        if s is None or not s.alive or not 0 <= new_len <= s.len:
            return ERR_ARG
        keep = _ceil_div(new_len, self.bs)
        for b in reversed(s.pt[keep:]):
            self.unref_block(b)
        del s.pt[keep:]
        s.len = new_len
        return OK

    def seq_truncate_batch(self, seqs, new_lens) -> int:
        """Truncate several sequences: every row is validated before any changes."""
        if len(seqs) != len(new_lens) or len(seqs) == 0:
            return ERR_ARG
        if len({id(s) for s in seqs}) != len(seqs):
            return ERR_ARG
        for s, n in zip(seqs, new_lens):
            if s is None or not s.alive or not 0 <= n <= s.len:
                return ERR_ARG
        for s, n in zip(seqs, new_lens):
            self.seq_truncate(s, n)
        return OK

    # ---- step calls (caller contract) ------------------------------------------
    def _ensure_one(self, s: SeqModel, n: int) -> int:
        if s is None or not s.alive or n <= 0:
            return ERR_ARG
        if s.len + n > s.max_tokens:
            return ERR_CAPACITY
        first = s.len // self.bs
        last = (s.len + n - 1) // self.bs
        cow = [k for k in range(first, min(last + 1, len(s.pt))) if self.refcnt[s.pt[k]] > 1]
        new = max(0, last + 1 - len(s.pt))
        if len(self.free) < len(cow) + new:
            return ERR_EXHAUSTED
        for k in cow:
            nb = self.alloc_block()
            self.unref_block(s.pt[k])
            s.pt[k] = nb
        while len(s.pt) < last + 1:
            s.pt.append(self.alloc_block())
        return OK

    def ensure_append(self, s: SeqModel, n: int) -> int:
        return self.ensure_append_batch([s], [n])

    def ensure_append_batch(self, seqs, ns) -> int:
        if len(seqs) != len(ns) or len(seqs) == 0:
            return ERR_ARG
        if len({id(s) for s in seqs}) != len(seqs):
            return ERR_ARG
        # all-or-nothing: run the batch on a copy, commit only if every row fits
        trial = copy.deepcopy(self)
        index = {id(s): i for i, s in enumerate(self.seqs)}
        for s, n in zip(seqs, ns):
            if s is None or not s.alive or id(s) not in index:
                return ERR_ARG
            rc = trial._ensure_one(trial.seqs[index[id(s)]], n)
            if rc != OK:
                return rc
        self.free, self.refcnt = trial.free, trial.refcnt
        for s, t in zip(self.seqs, trial.seqs):
            s.pt, s.len = t.pt, t.len
        return OK

    def advance(self, s: SeqModel, n: int) -> int:
        return self.advance_batch([s], [n])

    def advance_batch(self, seqs, ns) -> int:
        if len(seqs) != len(ns) or len(seqs) == 0:
            return ERR_ARG
        if len({id(s) for s in seqs}) != len(seqs):
            return ERR_ARG
        for s, n in zip(seqs, ns):
            if s is None or not s.alive or n <= 0:
                return ERR_ARG
            if s.len + n > s.max_tokens:
                return ERR_CAPACITY
            if s.len + n > len(s.pt) * self.bs:
                return ERR_SEQ
        for s, n in zip(seqs, ns):
            s.len += n
        return OK

    def can_append(self, s: SeqModel, n: int) -> int:
        """Reading 6: the rows [len, len+n) must lie in existing private blocks."""
        if s is None or not s.alive:
            return ERR_SEQ
        if n <= 0:
            return ERR_BAD_DIM
        if s.len + n > len(s.pt) * self.bs:
            return ERR_SEQ
        for k in range(s.len // self.bs, (s.len + n - 1) // self.bs + 1):
            if self.refcnt[s.pt[k]] != 1:
                return ERR_SEQ
        return OK

    # ---- invariants ------------------------------------------------------------
    def check_invariants(self, extra_refs=None) -> None:
        """Every block is either free (refcount 0) or referenced exactly
        refcount times by page tables plus ``extra_refs`` (ids the caller holds
        from alloc_block)."""
        count = [0] * self.n_blocks
        for s in self.seqs:
            for b in s.pt:
                count[b] += 1
        for b in (extra_refs or []):
            count[b] += 1
        free = set(self.free)
        assert len(free) == len(self.free), "block on the free list twice"
        for b in range(self.n_blocks):
            assert count[b] == self.refcnt[b], (b, count[b], self.refcnt[b])
            assert (b in free) == (self.refcnt[b] == 0), b


__all__ = ["PoolModel", "SeqModel", "OK", "ERR_BAD_DIM", "ERR_BAD_GQA", "ERR_SEQ",
           "ERR_EXHAUSTED", "ERR_CAPACITY", "ERR_ARG"]
