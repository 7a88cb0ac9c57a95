"""Fused append + decode vs the unfused path (append kernel, then attend).

The per-layer step appends the new K/V rows into their pages and then attends
over the sequence ("nx_f32_attn_paged.nx source", header comment and step 1
of nx_f32_attn_with_paged).  With fusion the decode kernel reads the new rows from K_new /
V_new, stores them into the pool and enters fresh pages into the device page
table.  Both paths must give the same bits: outputs, pool contents, page
tables.  Each case runs twice on identically built pools (same shuffled free
list, same seeded data), once per mode, and compares everything bit for bit.
"""
from __future__ import annotations

import pytest
import torch

import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool, bits_equal
from synth import workloads as wl

H, KV, HD = 32, 8, 128


@pytest.fixture
def fused_mode():
    old = pkv.pkv_get_fused_append()
    yield
    pkv.pkv_set_fused_append(old)


DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.float8_e4m3fn}


def _run(fused, lens, n_q, steps, n_layers=2, bs=16, seed=7, fork_tail=False, split=None,
         dtype="f32", kv_scale=1.0, heads=(H, KV)):
    """Build a pool, write seeded histories, then `steps` decode steps of n_q
    tokens per row.  Returns the per-(step, layer) outputs, the pool tensors,
    the host page tables and the launch counts of the steps per kind."""
    H, KV = heads
    pkv.pkv_set_fused_append(fused)
    old_split = pkv.pkv_get_split_keys()
    if split:
        pkv.check(pkv.pkv_set_split_keys(split))
    kv_dim = KV * HD
    max_tok = max(lens) + n_q * steps + 8
    n_blocks = sum((L + n_q * steps + bs) // bs + 2 for L in lens) + 16
    pool = GpuPool(n_blocks, n_layers, kv_dim, bs, max_seqs=2 * len(lens) + 2,
                   max_blocks=(max_tok + bs - 1) // bs + 1, shuffle_seed=seed,
                   dtype=DTYPES[dtype], kv_scale=kv_scale)
    try:
        seqs = []
        for r, L in enumerate(lens):
            s = pool.new_seq(max_tok)
            pool.grow(s, L)
            for layer in range(n_layers):
                pool.write_history(s, layer, wl.normal((L, kv_dim), seed + 10 * r + layer, "cuda"),
                                   wl.normal((L, kv_dim), seed + 10 * r + layer + 5, "cuda"))
            seqs.append(s)
        if fork_tail:
            # forks share the partial tail page: their first append copies it
            seqs = [pkv.pkv_seq_fork(s) for s in seqs]
        pkv.check(pkv.pkv_pool_flush(pool.p))
        torch.cuda.synchronize()
        outs = []
        nq = [n_q] * len(seqs)
        T = n_q * len(seqs)
        pkv.pkv_profile_reset()
        pkv.pkv_profile_enable(True)
        for step in range(steps):
            pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
            for layer in range(n_layers):
                base = seed + 1000 * step + 100 * layer
                Q = wl.normal((T, H * HD), base + 1, "cuda")
                Kn = wl.normal((T, kv_dim), base + 2, "cuda")
                Vn = wl.normal((T, kv_dim), base + 3, "cuda")
                out = torch.empty(T, H * HD, device="cuda")
                pkv.check(pkv.pkv_attn_batch(seqs, nq, Q, Kn, Vn, H, KV, HD, layer, 1,
                                             HD ** -0.5, out))
                outs.append(out)
            pkv.check(pkv.pkv_advance_batch(seqs, nq))
        torch.cuda.synchronize()
        pkv.pkv_profile_enable(False)
        counts = {k: pkv.pkv_profile_read(k)[1] for k in range(pkv.PKV_KERNEL_KINDS)}
        counts["work"] = pkv.pkv_pool_last_work(pool.p)
        pkv.check(pkv.pkv_sync_error(pool.p))
        # the device page table is checked through the steps themselves: every
        # page a step enters is read back through it by the next step
        pts = [pkv.pkv_seq_page_table(s) for s in seqs]
        return outs, pool.K.clone(), pool.V.clone(), pts, counts
    finally:
        pkv.pkv_profile_reset()
        pkv.pkv_set_split_keys(old_split)
        pool.close()


def _compare(a, b):
    outs_a, Ka, Va, pta, _ = a
    outs_b, Kb, Vb, ptb, _ = b
    assert len(outs_a) == len(outs_b)
    for i, (x, y) in enumerate(zip(outs_a, outs_b)):
        assert bits_equal(x, y), "output %d differs between fused and unfused" % i
    assert pta == ptb
    # NaN-filled pools: compare bit patterns, so untouched rows match too
    as_bytes = lambda t: t.contiguous().view(torch.uint8)  # noqa: E731
    assert torch.equal(as_bytes(Ka), as_bytes(Kb)) and torch.equal(as_bytes(Va), as_bytes(Vb)), \
        "pool contents differ"


@pytest.mark.gpu
def test_fused_append_is_bit_exact_across_pages_and_splits(fused_mode):
    # lengths at and around page (16) and split (1024) boundaries
    lens = [15, 16, 31, 1023, 1024, 2047, 100, 5]
    fused = _run(True, lens, 1, steps=3)
    plain = _run(False, lens, 1, steps=3)
    _compare(fused, plain)
    # the fused steps launched no append kernel; the unfused ones one per layer call
    assert fused[4][pkv.PKV_KERNEL_APPEND] == 0
    assert plain[4][pkv.PKV_KERNEL_APPEND] == 3 * 2
    assert fused[4][pkv.PKV_KERNEL_DECODE] == plain[4][pkv.PKV_KERNEL_DECODE] == 3 * 2
    assert fused[4]["work"]["fused_append"] == 1 and plain[4]["work"]["fused_append"] == 0


@pytest.mark.gpu
def test_fused_append_multi_query_rows_cross_a_split(fused_mode):
    # 3 new tokens per row (below the tensor-core threshold): rows at 1022 and
    # 2046 put their new positions on both sides of a split boundary
    lens = [1022, 2046, 40, 7]
    fused = _run(True, lens, 3, steps=2)
    plain = _run(False, lens, 3, steps=2)
    _compare(fused, plain)
    assert fused[4][pkv.PKV_KERNEL_APPEND] == 0


@pytest.mark.gpu
@pytest.mark.parametrize("bs", [4, 8], ids=["bs4", "bs8"])
def test_fused_append_small_pages(bs, fused_mode):
    # bs 4: tiles of 8 keys span pages (per-position lookups); bs 8: one page per tile
    lens = [3, 8, 33, 300]
    fused = _run(True, lens, 1, steps=3, bs=bs, split=64)
    plain = _run(False, lens, 1, steps=3, bs=bs, split=64)
    _compare(fused, plain)
    assert fused[4][pkv.PKV_KERNEL_APPEND] == 0


@pytest.mark.gpu
def test_fused_append_falls_back_on_copy_on_append(fused_mode):
    # forks of sequences with a partial tail page: the first append copies the
    # tail (old positions in a changed page), so that call runs unfused; the
    # later steps allocate fresh pages only and fuse again
    lens = [21, 50, 7]
    fused = _run(True, lens, 1, steps=3, fork_tail=True)
    plain = _run(False, lens, 1, steps=3, fork_tail=True)
    _compare(fused, plain)
    assert fused[4][pkv.PKV_KERNEL_APPEND] == 1
    assert plain[4][pkv.PKV_KERNEL_APPEND] == 3 * 2


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,kv_scale,heads", [("bf16", 1.0, (32, 8)), ("bf16", 1.0, (16, 8)),
                                                  ("fp8", 1.0, (32, 8)), ("fp8", 2.0, (64, 8))],
                         ids=["bf16-g4", "bf16-g2", "fp8-g4", "fp8-scale2-g8"])
def test_fused_append_narrow_pools(dtype, kv_scale, heads, fused_mode):
    """bf16 and fp8 pools: the narrow-pool decode kernel takes the append
    itself, rounding the new rows exactly as the append kernel does (fp8:
    e4m3 of x / scale, saturating); outputs, pool bytes and page tables equal
    the unfused path's."""
    lens = [15, 16, 31, 1023, 1024, 2047, 100, 5]
    fused = _run(True, lens, 1, steps=3, dtype=dtype, kv_scale=kv_scale, heads=heads)
    plain = _run(False, lens, 1, steps=3, dtype=dtype, kv_scale=kv_scale, heads=heads)
    _compare(fused, plain)
    assert fused[4][pkv.PKV_KERNEL_APPEND] == 0
    assert plain[4][pkv.PKV_KERNEL_APPEND] == 3 * 2
    assert fused[4]["work"]["fused_append"] == 1


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_fused_append_narrow_pools_multi_query_and_small_pages(dtype, fused_mode):
    # 3 new tokens per row on both sides of a split boundary; then block
    # size 4, where a 16- or 32-key tile spans several pages
    for kw in (dict(lens=[1022, 2046, 40, 7], n_q=3, steps=2),
               dict(lens=[3, 8, 33, 300], n_q=1, steps=3, bs=4, split=64)):
        lens, n_q, steps = kw.pop("lens"), kw.pop("n_q"), kw.pop("steps")
        fused = _run(True, lens, n_q, steps, dtype=dtype, **kw)
        plain = _run(False, lens, n_q, steps, dtype=dtype, **kw)
        _compare(fused, plain)
        assert fused[4][pkv.PKV_KERNEL_APPEND] == 0
