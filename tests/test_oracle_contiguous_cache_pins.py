"""Pins for the oracle's contiguous-cache twin and the pool model's batch
truncate (CPU only).

``oracle.ContiguousCache`` is the reference side of the gate ("nx_paged_kv_gate.nx
source", EQUIV section: a contiguous cache of max_seq rows per layer, appended
and attended by nx_f32_attn_with_cache, moved on by nx_f32_kv_cache_advance;
FORK section: both forks equal fresh replays of their histories; REWIND
section: truncating to the fork point and appending the other fork's rows
gives that fork's outputs).  What the class adds to ``oracle.attend`` is
bookkeeping -- where a round's rows land, which rows a call sees, what a fork
and a truncate keep -- so the battery below checks that bookkeeping against
histories the test builds on its own, by concatenating the gate's round
arrays:

* Q = 0 makes every score 0, so query i of a round returns the plain mean of
  the visible value rows 0 .. q_pos (q_pos = total_k - n_q + i, the
  offset-causal position of "nx_f32_attn_paged.nx source").  That mean is
  computed here with numpy from the concatenated rows, without attend.
* With the gate's own queries the outputs equal ``attend`` over the
  concatenated history (attend itself is pinned in test_oracle_pins.py).
* Fork, rewind and the checks' order of return codes, per the gate.

``test_cache_mutations_are_caught`` plants plausible mistakes in copies of
the class (append one row late, attend over the committed rows only, a fork
that shares its arrays, a truncate that keeps the length, every layer
written to layer 0, advance counted twice) and checks that the battery
rejects every one.

``PoolModel.seq_truncate_batch`` is pinned on hand-worked batches: a batch
whose last row is invalid changes nothing (every row is validated before any
changes), and a valid batch releases exactly the blocks past
ceil(new_len / bs), last block first, onto the LIFO free list.
"""
import copy
import json
import os

import numpy as np
import pytest

import oracle
from oracle.contiguous_cache import ContiguousCache, ERR_SEQ
from oracle.pool_model import PoolModel, OK, ERR_ARG
from synth import gate_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
G = json.load(open(os.path.join(GOLDEN, "gate_constants.json")))
NL, H, KV, HD = G["n_layers"], G["n_heads"], G["n_kv_heads"], G["head_dim"]
GROUP = H // KV
SCALE = G["scale"]
MAX_SEQ = 64


def _round(cc, Q, K, V, n, layer_data=None):
    """One gate round on a cache: append + attend on every layer, then
    advance.  layer_data(layer, K, V) may give each layer its own rows."""
    outs = []
    for layer in range(NL):
        k, v = (K, V) if layer_data is None else layer_data(layer, K, V)
        rc, out = cc.attn_with_cache(Q, k, v, n, H, KV, HD, layer, 1, SCALE)
        assert rc == 0, rc
        outs.append(out)
    cc.advance(n)
    return outs


def _mean_rows(V_hist, n_q):
    """Expected output for Q = 0: query i sees value rows 0 .. total_k - n_q + i
    of its kv head; every head of a group gets its kv head's mean."""
    total_k = V_hist.shape[0]
    Vh = V_hist.astype(np.float64).reshape(total_k, KV, HD)
    out = np.empty((n_q, H, HD))
    for i in range(n_q):
        vis = total_k - n_q + i + 1
        for h in range(H):
            out[i, h] = Vh[:vis, h // GROUP].mean(axis=0)
    return out.reshape(n_q, H * HD)


def _layer_shift(layer, K, V):
    # distinct data per layer, so that a layer mix-up shows
    return K + 3.0 * layer, V + 100.0 * layer


# ---------------------------------------------------------------------------
# the battery: each pin takes a class with ContiguousCache's API


def pin_rounds_q0_mean(CC):
    """EQUIV rounds (5, 1, 3 tokens, two layers with different rows) with
    Q = 0: each round's output is the mean of the visible value rows of the
    history built here by concatenation."""
    x = gate_inputs(G["seed"])
    cc = CC(NL, KV, MAX_SEQ, HD)
    hist_v = [[] for _ in range(NL)]
    for name, n in zip(("1", "2", "3"), G["rounds"]):
        Q = np.zeros((n, H * HD), np.float32)
        outs = _round(cc, Q, x["K" + name], x["V" + name], n, _layer_shift)
        for layer in range(NL):
            hist_v[layer].append(_layer_shift(layer, x["K" + name], x["V" + name])[1])
            exp = _mean_rows(np.concatenate(hist_v[layer]), n)
            np.testing.assert_allclose(outs[layer], exp, rtol=0, atol=1e-5)
    assert cc.seq_len == sum(G["rounds"])
    for layer in range(NL):
        k, v = cc.history(layer)
        assert np.array_equal(v, np.concatenate(hist_v[layer]))
        assert k.shape == (cc.seq_len, KV * HD)


def pin_rounds_vs_attend(CC):
    """EQUIV rounds with the gate's own queries: each round equals attend over
    the concatenated history, bit for bit."""
    x = gate_inputs(G["seed"])
    cc = CC(NL, KV, MAX_SEQ, HD)
    Ks, Vs = [], []
    for name, n in zip(("1", "2", "3"), G["rounds"]):
        Q, K, V = x["Q" + name], x["K" + name], x["V" + name]
        outs = _round(cc, Q, K, V, n)
        Ks.append(K)
        Vs.append(V)
        Kh, Vh = np.concatenate(Ks), np.concatenate(Vs)
        rc, exp = oracle.attend(Q, Kh, Vh, n, Kh.shape[0], H, KV, HD, 1, SCALE)
        assert rc == 0
        for layer in range(NL):
            assert np.array_equal(outs[layer], exp)


def pin_fork_replay(CC):
    """FORK: fork after the 5-token prefill; fork A appends (QA, KA, VA), then
    fork B appends (QB, KB, VB).  Each fork's outputs equal a fresh cache that
    replays its history, and B's rows never reach A's history."""
    x = gate_inputs(G["seed"])
    n0, nd = G["fork_after"], G["diverge"]
    a = CC(NL, KV, MAX_SEQ, HD)
    _round(a, x["Q1"], x["K1"], x["V1"], n0)
    b = a.fork()
    outA = _round(a, x["QA"], x["KA"], x["VA"], nd)
    outB = _round(b, x["QB"], x["KB"], x["VB"], nd)
    for side, outs in (("A", outA), ("B", outB)):
        fresh = CC(NL, KV, MAX_SEQ, HD)
        _round(fresh, x["Q1"], x["K1"], x["V1"], n0)
        ref = _round(fresh, x["Q" + side], x["K" + side], x["V" + side], nd)
        for layer in range(NL):
            assert np.array_equal(outs[layer], ref[layer])
    # one more decode row on A with Q = 0: the mean over A's own history
    probe_k = np.zeros((1, KV * HD), np.float32)
    probe_v = np.full((1, KV * HD), 2.0, np.float32)
    outs = _round(a, np.zeros((1, H * HD), np.float32), probe_k, probe_v, 1)
    exp = _mean_rows(np.concatenate([x["V1"], x["VA"], probe_v]), 1)
    for layer in range(NL):
        np.testing.assert_allclose(outs[layer], exp, rtol=0, atol=1e-5)
    assert a.seq_len == n0 + nd + 1 and b.seq_len == n0 + nd


def pin_rewind(CC):
    """REWIND: fork A truncated to the fork point and fed B's rows answers
    exactly as fork B did."""
    x = gate_inputs(G["seed"])
    n0, nd = G["fork_after"], G["diverge"]
    a = CC(NL, KV, MAX_SEQ, HD)
    _round(a, x["Q1"], x["K1"], x["V1"], n0)
    b = a.fork()
    _round(a, x["QA"], x["KA"], x["VA"], nd)
    outB = _round(b, x["QB"], x["KB"], x["VB"], nd)
    a.truncate(G["truncate_to"])
    assert a.seq_len == G["truncate_to"]
    outR = _round(a, x["QB"], x["KB"], x["VB"], nd)
    for layer in range(NL):
        assert np.array_equal(outR[layer], outB[layer])
    with pytest.raises(ValueError):
        a.truncate(a.seq_len + 1)


def pin_checks(CC):
    """The argument checks of nx_f32_attn_with_paged, in order: sizes -> 1,
    grouping -> 2, storage (layer, room, shape) -> 3; a rejected call leaves
    the history as it was."""
    x = gate_inputs(G["seed"])
    cc = CC(NL, KV, 8, HD)
    Q, K, V = x["Q1"], x["K1"], x["V1"]
    assert cc.attn_with_cache(Q, K, V, 0, H, KV, HD, 0, 1, SCALE)[0] == 1
    assert cc.attn_with_cache(Q, K, V, 5, 0, KV, HD, 0, 1, SCALE)[0] == 1
    assert cc.attn_with_cache(Q, K, V, 5, 3, KV, HD, 0, 1, SCALE)[0] == 2
    assert cc.attn_with_cache(Q, K, V, 5, H, KV, HD, NL, 1, SCALE)[0] == ERR_SEQ
    _round(cc, Q, K, V, 5)
    big = np.zeros((4, KV * HD), np.float32)
    assert cc.attn_with_cache(np.zeros((4, H * HD), np.float32), big, big, 4, H, KV, HD, 0, 1,
                              SCALE)[0] == ERR_SEQ
    assert cc.seq_len == 5
    assert np.array_equal(cc.history(0)[1], V)


BATTERY = [pin_rounds_q0_mean, pin_rounds_vs_attend, pin_fork_replay, pin_rewind, pin_checks]


@pytest.mark.parametrize("pin", BATTERY, ids=lambda f: f.__name__)
def test_contiguous_cache_pins(pin):
    pin(ContiguousCache)


# ---------------------------------------------------------------------------
# planted mistakes: each copy of the class differs from the oracle's in one
# plausible way, and the battery must reject it


class _AppendLate(ContiguousCache):
    """Writes a round's rows one position late (a hole at seq_len)."""

    def attn_with_cache(self, Q, K_new, V_new, n_tokens, n_heads, n_kv_heads, head_dim, layer,
                        causal, scale):
        if n_tokens <= 0 or n_heads <= 0 or n_kv_heads <= 0 or head_dim <= 0:
            return 1, None
        if n_heads % n_kv_heads != 0:
            return 2, None
        if not 0 <= layer < self.n_layers or self.seq_len + n_tokens + 1 > self.max_seq:
            return ERR_SEQ, None
        s = self.seq_len + 1
        self.K[layer, s:s + n_tokens] = np.asarray(K_new, np.float32).reshape(n_tokens, -1)
        self.V[layer, s:s + n_tokens] = np.asarray(V_new, np.float32).reshape(n_tokens, -1)
        total_k = self.seq_len + n_tokens
        return oracle.attend(Q, self.K[layer, :total_k], self.V[layer, :total_k], n_tokens,
                             total_k, n_heads, n_kv_heads, head_dim, causal, scale)


class _SliceCommitted(ContiguousCache):
    """Attends over the committed rows only (slice ends at seq_len)."""

    def attn_with_cache(self, Q, K_new, V_new, n_tokens, n_heads, n_kv_heads, head_dim, layer,
                        causal, scale):
        if n_tokens <= 0 or n_heads <= 0 or n_kv_heads <= 0 or head_dim <= 0:
            return 1, None
        if n_heads % n_kv_heads != 0:
            return 2, None
        if not 0 <= layer < self.n_layers or self.seq_len + n_tokens > self.max_seq:
            return ERR_SEQ, None
        s = self.seq_len
        self.K[layer, s:s + n_tokens] = np.asarray(K_new, np.float32).reshape(n_tokens, -1)
        self.V[layer, s:s + n_tokens] = np.asarray(V_new, np.float32).reshape(n_tokens, -1)
        total_k = s + n_tokens
        return oracle.attend(Q, self.K[layer, :s], self.V[layer, :s], n_tokens, total_k,
                             n_heads, n_kv_heads, head_dim, causal, scale)


class _ShallowFork(ContiguousCache):
    """A fork that shares the parent's K/V stripes."""

    def fork(self):
        return copy.copy(self)


class _TruncateKeepsLength(ContiguousCache):
    def truncate(self, new_len):
        if not 0 <= new_len <= self.seq_len:
            raise ValueError("truncate outside [0, seq_len]")


class _OneLayer(ContiguousCache):
    """Every layer's rows go to (and are read from) layer 0."""

    def attn_with_cache(self, Q, K_new, V_new, n_tokens, n_heads, n_kv_heads, head_dim, layer,
                        causal, scale):
        return super().attn_with_cache(Q, K_new, V_new, n_tokens, n_heads, n_kv_heads, head_dim,
                                       0 if 0 <= layer < self.n_layers else layer, causal, scale)


class _AdvanceTwice(ContiguousCache):
    def advance(self, n):
        self.seq_len += 2 * n if self.seq_len + 2 * n <= self.max_seq else n


MUTANTS = [_AppendLate, _SliceCommitted, _ShallowFork, _TruncateKeepsLength, _OneLayer,
           _AdvanceTwice]


def _battery_rejects(CC):
    for pin in BATTERY:
        try:
            pin(CC)
        except (AssertionError, ValueError, IndexError):
            return True
    return False


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda c: c.__name__)
def test_cache_mutations_are_caught(mutant):
    assert _battery_rejects(mutant), mutant.__doc__ or mutant.__name__


# ---------------------------------------------------------------------------
# PoolModel.seq_truncate_batch


def _grown_pool():
    """Three sequences at block size 4: lengths 10, 7 and 13 (3, 2 and 4
    blocks), taken from a fresh pool in batch order."""
    p = PoolModel(16, 1, 16, 4, 8, 8)
    seqs = [p.seq_new(32) for _ in range(3)]
    for s, n in zip(seqs, (10, 7, 13)):
        assert p.ensure_append(s, n) == OK and p.advance(s, n) == OK
    return p, seqs


def _state(p, seqs):
    return (list(p.free), list(p.refcnt), [(s.len, list(s.pt)) for s in seqs])


def test_truncate_batch_hand_worked():
    p, (a, b, c) = _grown_pool()
    # fresh pops ascend: a holds 0..2, b 3..4, c 5..8; 7 blocks stay free
    assert (a.pt, b.pt, c.pt) == ([0, 1, 2], [3, 4], [5, 6, 7, 8])
    assert p.seq_truncate_batch([a, b, c], [5, 7, 0]) == OK
    # a keeps ceil(5/4) = 2 blocks, b all 2, c none
    assert (a.len, a.pt) == (5, [0, 1])
    assert (b.len, b.pt) == (7, [3, 4])
    assert (c.len, c.pt) == (0, [])
    # released in batch order, each sequence's last block first: 2, then 8, 7, 6, 5;
    # the next pops take the latest release first
    assert [p.alloc_block() for _ in range(5)] == [5, 6, 7, 8, 2]
    p.check_invariants(extra_refs=[5, 6, 7, 8, 2])


@pytest.mark.parametrize("bad", [
    ([5, 7, 14], "last row grows"),
    ([5, 7, -1], "last row negative"),
    ([11, 3, 4], "first row grows"),
])
def test_truncate_batch_is_all_or_nothing(bad):
    lens, _ = bad
    p, seqs = _grown_pool()
    snap = _state(p, seqs)
    assert p.seq_truncate_batch(seqs, lens) == ERR_ARG
    assert _state(p, seqs) == snap


def test_truncate_batch_rejects_duplicates_and_mismatch():
    p, (a, b, c) = _grown_pool()
    snap = _state(p, [a, b, c])
    assert p.seq_truncate_batch([a, b, a], [1, 1, 1]) == ERR_ARG
    assert p.seq_truncate_batch([a, b], [1]) == ERR_ARG
    assert p.seq_truncate_batch([], []) == ERR_ARG
    assert _state(p, [a, b, c]) == snap


class _TruncateAsYouGo(PoolModel):
    """Applies each row as it validates it (not all-or-nothing)."""

    def seq_truncate_batch(self, seqs, new_lens):
        for s, n in zip(seqs, new_lens):
            if self.seq_truncate(s, n) != OK:
                return ERR_ARG
        return OK


def test_truncate_batch_mutation_is_caught():
    p = _TruncateAsYouGo(16, 1, 16, 4, 8, 8)
    seqs = [p.seq_new(32) for _ in range(3)]
    for s, n in zip(seqs, (10, 7, 13)):
        assert p.ensure_append(s, n) == OK and p.advance(s, n) == OK
    snap = _state(p, seqs)
    assert p.seq_truncate_batch(seqs, [5, 7, 14]) == ERR_ARG
    assert _state(p, seqs) != snap
