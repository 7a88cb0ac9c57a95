"""Operand-image cache (pkv_pool_set_image_cache; not on the pages).

Every case runs the same calls on two pools with the same contents and block
layout, one with the cache on and one with it off: the images a cached call
reads are the bits the split pass would write again, so the outputs must be
equal bit for bit.  The cached pool's work counters show which tiles came from
the cache; a few outputs are also checked against the oracle.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool, assert_close, bits_equal

H, KV, HD, BS = 32, 8, 128, 16
KV_DIM, Q_DIM = KV * HD, H * HD
SCALE = float(np.float32(1.0 / math.sqrt(HD)))
CACHE_BYTES = 512 << 20


class Twin:
    """Two pools driven through the same calls; pool 0 has the image cache."""

    def __init__(self, n_blocks, max_tokens, n_seqs=1, cache_bytes=CACHE_BYTES):
        self.pools = [GpuPool(n_blocks, 1, KV_DIM, BS, max_seqs=n_seqs + 8,
                              max_blocks=-(-max_tokens // BS) + 1, shuffle_seed=3) for _ in range(2)]
        pkv.check(pkv.pkv_pool_set_image_cache(self.pools[0].p, cache_bytes))

    def close(self):
        for p in self.pools:
            p.close()

    def attend(self, seqs, nq, Q, K, V):
        outs = []
        for p, ss in zip(self.pools, seqs):
            pkv.check(pkv.pkv_ensure_append_batch(ss, nq))
            out = torch.empty(Q.shape[0], Q_DIM, device="cuda")
            pkv.check(pkv.pkv_attn_batch(ss, nq, Q, K, V, H, KV, HD, 0, 1, SCALE, out))
            pkv.check(pkv.pkv_advance_batch(ss, nq))
            p.check_no_device_error()
            outs.append(out)
        torch.cuda.synchronize()
        assert bits_equal(outs[0], outs[1]), "cached and uncached outputs differ"
        return outs[0], pkv.pkv_pool_last_work(self.pools[0].p)


def _rand(n, d, g):
    return torch.randn(n, d, generator=g, device="cuda")


@pytest.mark.gpu
def test_chunked_prefill_reuses_earlier_tiles():
    past, chunk, n_chunks = 1000, 128, 4
    g = torch.Generator(device="cuda").manual_seed(1)
    tw = Twin(-(-(past + chunk * n_chunks) // BS) + 8, past + chunk * n_chunks + 1)
    try:
        seqs = [[p.new_seq(past + chunk * n_chunks)] for p in tw.pools]
        Kh, Vh = _rand(past, KV_DIM, g), _rand(past, KV_DIM, g)
        for p, ss in zip(tw.pools, seqs):
            p.grow(ss[0], past)
            p.write_history(ss[0], 0, Kh, Vh)
        Kall, Vall = [Kh.cpu().numpy()], [Vh.cpu().numpy()]
        for c in range(n_chunks):
            Q, K, V = _rand(chunk, Q_DIM, g), _rand(chunk, KV_DIM, g), _rand(chunk, KV_DIM, g)
            out, wk = tw.attend(seqs, [chunk], Q, K, V)
            L = past + chunk * (c + 1)
            n_tiles = -(-L // 64)
            assert wk["image_hits"] + wk["image_builds"] == n_tiles
            # the tiles wholly below the pages written since the last call are reused
            first_written = (past + chunk * c) // BS * BS
            assert wk["image_hits"] == (0 if c == 0 else first_written // 64), (c, wk)
            Kall.append(K.cpu().numpy())
            Vall.append(V.cpu().numpy())
            Kf, Vf = np.concatenate(Kall), np.concatenate(Vall)
            for i in (0, chunk - 1):
                rc, ref = oracle.attend(Q[i:i + 1].cpu().numpy(), Kf, Vf, 1, L - chunk + i + 1, H, KV, HD, 1, SCALE)
                assert rc == 0
                assert_close(out[i:i + 1].cpu().numpy(), ref, np.abs(Vf).max(), "chunk %d query %d" % (c, i))
    finally:
        tw.close()


@pytest.mark.gpu
def test_rewrite_after_truncate_is_seen():
    # rows rewritten at the same positions (truncate, then append other
    # values) get new page generations: the cached pool must not reuse images
    # of the old rows
    past, chunk = 512, 96
    g = torch.Generator(device="cuda").manual_seed(2)
    tw = Twin(64, past + 2 * chunk + 1)
    try:
        seqs = [[p.new_seq(past + 2 * chunk)] for p in tw.pools]
        Kh, Vh = _rand(past, KV_DIM, g), _rand(past, KV_DIM, g)
        for p, ss in zip(tw.pools, seqs):
            p.grow(ss[0], past)
            p.write_history(ss[0], 0, Kh, Vh)
        for rnd in range(3):
            Q, K, V = _rand(chunk, Q_DIM, g), _rand(chunk, KV_DIM, g), _rand(chunk, KV_DIM, g)
            tw.attend(seqs, [chunk], Q, K, V)
            Q2 = _rand(chunk, Q_DIM, g)
            _, wk = tw.attend(seqs, [chunk], Q2, _rand(chunk, KV_DIM, g), _rand(chunk, KV_DIM, g))
            assert wk["image_hits"] > 0
            for ss in seqs:
                pkv.check(pkv.pkv_seq_truncate(ss[0], past))
    finally:
        tw.close()


@pytest.mark.gpu
def test_direct_write_then_reset():
    past, chunk = 700, 64
    g = torch.Generator(device="cuda").manual_seed(3)
    tw = Twin(64, past + chunk + 1)
    try:
        seqs = [[p.new_seq(past + chunk)] for p in tw.pools]
        Kh, Vh = _rand(past, KV_DIM, g), _rand(past, KV_DIM, g)
        for p, ss in zip(tw.pools, seqs):
            p.grow(ss[0], past)
            p.write_history(ss[0], 0, Kh, Vh)
        Q, K, V = _rand(chunk, Q_DIM, g), _rand(chunk, KV_DIM, g), _rand(chunk, KV_DIM, g)
        tw.attend(seqs, [chunk], Q, K, V)
        for ss in seqs:
            pkv.check(pkv.pkv_seq_truncate(ss[0], past))
        # history rewritten behind the library's back, then the cache is reset
        Kh2, Vh2 = _rand(past, KV_DIM, g), _rand(past, KV_DIM, g)
        for p, ss in zip(tw.pools, seqs):
            p.write_history(ss[0], 0, Kh2, Vh2)
        pkv.check(pkv.pkv_pool_set_image_cache(tw.pools[0].p, CACHE_BYTES))
        _, wk = tw.attend(seqs, [chunk], Q, K, V)
        assert wk["image_hits"] == 0
    finally:
        tw.close()


@pytest.mark.gpu
def test_shared_prefix_steps_reuse_prefix_images():
    prefix, n_f = 2560, 20
    g = torch.Generator(device="cuda").manual_seed(4)
    tw = Twin(prefix // BS + 4 * n_f + 16, prefix + 40, n_seqs=n_f + 2)
    try:
        Kp, Vp = _rand(prefix, KV_DIM, g), _rand(prefix, KV_DIM, g)
        forks = []
        for p in tw.pools:
            root = p.new_seq(prefix + 40)
            p.grow(root, prefix)
            p.write_history(root, 0, Kp, Vp)
            forks.append([pkv.pkv_seq_fork(root) for _ in range(n_f)])
        for step in range(3):
            Q, K, V = _rand(n_f, Q_DIM, g), _rand(n_f, KV_DIM, g), _rand(n_f, KV_DIM, g)
            _, wk = tw.attend(forks, [1] * n_f, Q, K, V)
            assert wk["prefix_tiles"] > 0
            assert wk["image_hits"] == (0 if step == 0 else prefix // 64), (step, wk)
    finally:
        tw.close()


@pytest.mark.gpu
def test_cache_smaller_than_a_call_builds_everything():
    past, chunk = 1500, 64
    g = torch.Generator(device="cuda").manual_seed(5)
    one_slot = KV * 128 * 1024
    tw = Twin(128, past + 2 * chunk + 1, cache_bytes=4 * one_slot)
    try:
        seqs = [[p.new_seq(past + 2 * chunk)] for p in tw.pools]
        Kh, Vh = _rand(past, KV_DIM, g), _rand(past, KV_DIM, g)
        for p, ss in zip(tw.pools, seqs):
            p.grow(ss[0], past)
            p.write_history(ss[0], 0, Kh, Vh)
        for _ in range(2):
            _, wk = tw.attend(seqs, [chunk], _rand(chunk, Q_DIM, g), _rand(chunk, KV_DIM, g),
                              _rand(chunk, KV_DIM, g))
            assert wk["image_hits"] == 0 and wk["image_builds"] > 4
    finally:
        tw.close()


@pytest.mark.gpu
def test_image_cache_argument_checks():
    pool = GpuPool(8, 1, KV_DIM, BS)
    try:
        assert pkv.pkv_pool_set_image_cache(pool.p, -1) == pkv.PKV_ERR_ARG
        assert pkv.pkv_pool_set_image_cache(None, 1 << 20) == pkv.PKV_ERR_ARG
        assert pkv.pkv_pool_set_image_cache(pool.p, 0) == pkv.PKV_OK
        assert pkv.pkv_pool_set_image_cache(pool.p, 1 << 20) == pkv.PKV_OK
    finally:
        pool.close()


@pytest.mark.gpu
def test_two_layers_and_copy_on_append():
    # forks of an unaligned prefix: the first append copies the shared tail
    # page (a new block, new generation) in each fork; two layers keep
    # separate images of the same pages
    prefix, n_f, chunk, L = 1000, 3, 80, 2
    g = torch.Generator(device="cuda").manual_seed(6)
    pools = [GpuPool(prefix // BS + 24 * n_f + 16, L, KV_DIM, BS, max_seqs=n_f + 4,
                     max_blocks=(prefix + 3 * chunk) // BS + 2, shuffle_seed=7) for _ in range(2)]
    try:
        pkv.check(pkv.pkv_pool_set_image_cache(pools[0].p, CACHE_BYTES))
        hist = [(_rand(prefix, KV_DIM, g), _rand(prefix, KV_DIM, g)) for _ in range(L)]
        forks = []
        for p in pools:
            root = p.new_seq(prefix + 3 * chunk)
            p.grow(root, prefix)
            for layer in range(L):
                p.write_history(root, layer, *hist[layer])
            forks.append([pkv.pkv_seq_fork(root) for _ in range(n_f)])
        for c in range(3):
            nq = [chunk] * n_f
            for p, ff in zip(pools, forks):
                pkv.check(pkv.pkv_ensure_append_batch(ff, nq))
            for layer in range(L):
                Q = _rand(n_f * chunk, Q_DIM, g)
                K, V = _rand(n_f * chunk, KV_DIM, g), _rand(n_f * chunk, KV_DIM, g)
                outs = []
                for p, ff in zip(pools, forks):
                    out = torch.empty(n_f * chunk, Q_DIM, device="cuda")
                    pkv.check(pkv.pkv_attn_batch(ff, nq, Q, K, V, H, KV, HD, layer, 1, SCALE, out))
                    p.check_no_device_error()
                    outs.append(out)
                torch.cuda.synchronize()
                assert bits_equal(outs[0], outs[1]), "chunk %d layer %d" % (c, layer)
                wk = pkv.pkv_pool_last_work(pools[0].p)
                if c > 0:
                    assert wk["image_hits"] > 0, (c, layer, wk)
            for p, ff in zip(pools, forks):
                pkv.check(pkv.pkv_advance_batch(ff, nq))
    finally:
        for p in pools:
            p.close()
