"""Placement of the tensor-core prefill tiles (pkv_set_prefill_pairing).

A CTA of the tensor-core kernel runs two 128-row query tiles of one row and
key split side by side (two softmax chains sharing each K/V tile), or one
tile when its partner is absent.  Each chain's arithmetic is its own, so a
batch must return the same bits whether every tile runs alone (mode 0), in
pairs (mode 1) or in the balanced placement (mode 2, the default), and match
the oracle.  The batch has rows with odd tile counts (a tile without a
partner) and, with 64-key decode splits (prefill splits of 1024 keys), pairs
whose two tiles have different split counts (a split where only one of them
is present).
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool, assert_close, bits_equal

H, KV, HD = 32, 8, 128
ROWS = [(2900, 256), (2500, 200), (3100, 256), (1800, 96), (2000, 33)]  # (past, n_q)


def test_prefill_pairing_mode_range():
    old = pkv.pkv_get_prefill_pairing()
    try:
        assert pkv.pkv_set_prefill_pairing(3) == pkv.PKV_ERR_ARG
        assert pkv.pkv_set_prefill_pairing(-1) == pkv.PKV_ERR_ARG
        assert pkv.pkv_get_prefill_pairing() == old
        for mode in (0, 1, 2):
            assert pkv.pkv_set_prefill_pairing(mode) == pkv.PKV_OK
            assert pkv.pkv_get_prefill_pairing() == mode
    finally:
        pkv.pkv_set_prefill_pairing(old)


@pytest.mark.gpu
def test_prefill_pairing_modes_same_bits():
    rng = np.random.default_rng(zlib.crc32(b"pairing"))
    kv_dim, bs = KV * HD, 16
    scale = float(np.float32(1.0 / math.sqrt(HD)))
    hist = [(rng.standard_normal((p + n, kv_dim)).astype(np.float32),
             rng.standard_normal((p + n, kv_dim)).astype(np.float32)) for p, n in ROWS]
    Q = rng.standard_normal((sum(n for _, n in ROWS), H * HD)).astype(np.float32)
    blocks = sum(-(-(p + n) // bs) for p, n in ROWS)
    old_mode, old_split = pkv.pkv_get_prefill_pairing(), pkv.pkv_get_split_keys()
    outs, ctas, tiles = {}, {}, {}
    try:
        pkv.check(pkv.pkv_set_split_keys(64))
        for mode in (2, 1, 0):
            pool = GpuPool(blocks + 8, 1, kv_dim, bs, max_seqs=8, max_blocks=blocks, shuffle_seed=11)
            try:
                seqs = []
                for (p, n), (K, V) in zip(ROWS, hist):
                    s = pool.new_seq(p + n)
                    pool.grow(s, p)
                    pool.write_history(s, 0, torch.from_numpy(K[:p]), torch.from_numpy(V[:p]))
                    seqs.append(s)
                n_q = [n for _, n in ROWS]
                pkv.check(pkv.pkv_ensure_append_batch(seqs, n_q))
                Kn = np.concatenate([K[p:] for (p, _), (K, _) in zip(ROWS, hist)])
                Vn = np.concatenate([V[p:] for (p, _), (_, V) in zip(ROWS, hist)])
                Qd, Kd, Vd = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (Q, Kn, Vn))
                out = torch.empty(Q.shape[0], H * HD, device="cuda")
                pkv.check(pkv.pkv_set_prefill_pairing(mode))
                pkv.check(pkv.pkv_attn_batch(seqs, n_q, Qd, Kd, Vd, H, KV, HD, 0, 1, scale, out))
                pool.check_no_device_error()
                wk = pkv.pkv_pool_last_work(pool.p)
                outs[mode], ctas[mode], tiles[mode] = out, wk["prefill_ctas"], wk["prefill_tiles"]
            finally:
                pool.close()
    finally:
        pkv.pkv_set_prefill_pairing(old_mode)
        pkv.pkv_set_split_keys(old_split)
    assert tiles[0] == tiles[1] == tiles[2] > 0
    assert ctas[0] == tiles[0] * KV                      # one tile per CTA
    assert ctas[1] < ctas[0]                             # pairs
    assert ctas[1] <= ctas[2] <= ctas[0], ctas           # some pairs split, at most all
    assert bits_equal(outs[1], outs[0]), "pairs != single tiles"
    assert bits_equal(outs[2], outs[0]), "balanced placement != single tiles"
    # the oracle on the row with a tile without a partner and on the two-tile row
    q0 = 0
    for (p, n), (K, V) in zip(ROWS, hist):
        if (p, n) in ((2500, 200), (2000, 33)):
            rc, exp = oracle.attend(Q[q0:q0 + n], K, V, n, p + n, H, KV, HD, 1, scale)
            assert rc == 0
            assert_close(outs[2][q0:q0 + n].cpu().numpy(), exp, np.abs(V).max(), "row %d" % n)
        q0 += n
