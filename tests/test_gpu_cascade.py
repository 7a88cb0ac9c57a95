"""Shared-prefix (cascade) decode against the oracle.

Forks share their prefix pages ("nx_paged_kv_gate.nx source", FORK section:
the fork holds its parent's pages and each shared page's refcount reads 2).  A batch with a run of 16 or
more one-query rows over common prefix pages attends those keys once for the
run (a tensor-core pass over the stacked queries) and each row's own keys in
the decode kernel, then merges the two.  Every row is checked against the
oracle on histories built from the generator's draws (the prefix written into
the pool with torch indexing, each fork's own rows fed as K_new / V_new), and
the cascade run against the same batch with the cascade switched off.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool, assert_close
from synth import workloads as wl


@pytest.fixture
def cascade_mode():
    old = pkv.pkv_get_cascade()
    yield
    pkv.pkv_set_cascade(old)


def _forks_then_decode(H, KV, prefix, div, extra=(), cascade=True, seed=5, bs=16):
    """A root of `prefix` tokens, one fork per entry of `div` appending that
    many own tokens, plus unrelated sequences of the lengths in `extra`; then
    one decode step over [forks..., extras...].  Returns (outputs, expected,
    per-kind launch counts of the decode step, vmax per row)."""
    hd = 128
    kv_dim, q_dim = KV * hd, H * hd
    scale = float(np.float32(1.0 / math.sqrt(hd)))
    max_tok = prefix + max(list(div) + [0]) + max(list(extra) + [0]) + 4
    need = (prefix // bs + 2) + sum(max(d, 1) // bs + 3 for d in div) + sum(e // bs + 3 for e in extra)
    pool = GpuPool(need + 16, 1, kv_dim, bs, max_seqs=len(div) + len(extra) + 4,
                   max_blocks=max_tok // bs + 2, shuffle_seed=seed)
    pkv.pkv_set_cascade(cascade)
    try:
        rng = np.random.default_rng(seed)
        root = pool.new_seq(max_tok)
        Kp = rng.standard_normal((prefix, kv_dim)).astype(np.float32)
        Vp = rng.standard_normal((prefix, kv_dim)).astype(np.float32)
        pool.grow(root, prefix)
        pool.write_history(root, 0, torch.from_numpy(Kp), torch.from_numpy(Vp))
        forks = [pkv.pkv_seq_fork(root) for _ in div]
        hist = {}
        # each fork's own rows go through the library (as K_new / V_new)
        T = int(sum(div))
        Kd = rng.standard_normal((T, kv_dim)).astype(np.float32)
        Vd = rng.standard_normal((T, kv_dim)).astype(np.float32)
        Qd = rng.standard_normal((T, q_dim)).astype(np.float32)
        pkv.check(pkv.pkv_ensure_append_batch(forks, list(div)))
        tmp = torch.empty(T, q_dim, device="cuda")
        pkv.check(pkv.pkv_attn_batch(forks, list(div), torch.from_numpy(Qd).cuda(),
                                     torch.from_numpy(Kd).cuda(), torch.from_numpy(Vd).cuda(),
                                     H, KV, hd, 0, 1, scale, tmp))
        pkv.check(pkv.pkv_advance_batch(forks, list(div)))
        o = 0
        for f, d in zip(forks, div):
            hist[f] = (np.concatenate([Kp, Kd[o:o + d]]), np.concatenate([Vp, Vd[o:o + d]]))
            o += d
        others = []
        for L in extra:
            s = pool.new_seq(max_tok)
            Ke = rng.standard_normal((L, kv_dim)).astype(np.float32)
            Ve = rng.standard_normal((L, kv_dim)).astype(np.float32)
            pool.grow(s, L)
            pool.write_history(s, 0, torch.from_numpy(Ke), torch.from_numpy(Ve))
            hist[s] = (Ke, Ve)
            others.append(s)
        seqs = forks + others
        M = len(seqs)
        Q = rng.standard_normal((M, q_dim)).astype(np.float32)
        Kn = rng.standard_normal((M, kv_dim)).astype(np.float32)
        Vn = rng.standard_normal((M, kv_dim)).astype(np.float32)
        pkv.check(pkv.pkv_ensure_append_batch(seqs, [1] * M))
        pkv.check(pkv.pkv_pool_flush(pool.p))
        torch.cuda.synchronize()
        out = torch.empty(M, q_dim, device="cuda")
        pkv.pkv_profile_reset()
        pkv.pkv_profile_enable(True)
        pkv.check(pkv.pkv_attn_batch(seqs, [1] * M, torch.from_numpy(Q).cuda(),
                                     torch.from_numpy(Kn).cuda(), torch.from_numpy(Vn).cuda(),
                                     H, KV, hd, 0, 1, scale, out))
        torch.cuda.synchronize()
        pkv.pkv_profile_enable(False)
        counts = {k: pkv.pkv_profile_read(k)[1] for k in range(pkv.PKV_KERNEL_KINDS)}
        counts["work"] = pkv.pkv_pool_last_work(pool.p)
        pool.check_no_device_error()
        got = out.cpu().numpy()
        exp, vmax = [], []
        for r, s in enumerate(seqs):
            Kh, Vh = hist[s]
            Kf = np.concatenate([Kh, Kn[r:r + 1]])
            Vf = np.concatenate([Vh, Vn[r:r + 1]])
            rc, ref = oracle.attend(Q[r:r + 1], Kf, Vf, 1, Kf.shape[0], H, KV, hd, 1, scale)
            assert rc == 0
            exp.append(ref)
            vmax.append(float(np.abs(Vf).max()))
        return got, exp, counts, vmax
    finally:
        pkv.pkv_profile_reset()
        pool.close()


def _check_all(got, exp, vmax, what):
    for r, (e, v) in enumerate(zip(exp, vmax)):
        assert_close(got[r:r + 1], e, v, "%s row %d" % (what, r))


@pytest.mark.gpu
@pytest.mark.parametrize("H,KV", [(32, 8), (64, 8), (8, 8)], ids=["g4", "g8", "g1"])
def test_cascade_every_fork_matches_oracle(H, KV, cascade_mode):
    rng = np.random.default_rng(3)
    div = [int(x) for x in rng.integers(1, 40, size=40)]
    got, exp, counts, vmax = _forks_then_decode(H, KV, 3000, div)
    _check_all(got, exp, vmax, "cascade")
    # the shared prefix ran as one tensor-core pass over the whole pages
    assert counts[pkv.PKV_KERNEL_PREFILL] == 1
    Lp = (3000 // 16) * 16
    work = counts["work"]
    assert work["prefix_pairs"] == len(div) * Lp
    tq = 128 // (H // KV)
    sp = work["prefix_split_keys"]
    assert sp > 0 and sp % 64 == 0 and sp <= -(-Lp // 64) * 64
    assert work["prefix_tiles"] == -(-len(div) // tq) * -(-Lp // sp)
    assert work["decode_units"] == len(div) and work["merge_items"] == len(div)
    off, exp2, counts2, _ = _forks_then_decode(H, KV, 3000, div, cascade=False)
    assert counts2[pkv.PKV_KERNEL_PREFILL] == 0
    for r in range(len(div)):
        assert np.max(np.abs(got[r] - off[r])) <= 2e-5 * vmax[r] + 2e-6


@pytest.mark.gpu
def test_cascade_mixed_batch(cascade_mode):
    # forks with prefixes that end inside, on and past a page boundary, and
    # unrelated rows after them: only the forks form the group
    for prefix in (2047 + 16, 4096, 5000):
        div = [1 + (7 * i) % 23 for i in range(20)]
        got, exp, counts, vmax = _forks_then_decode(32, 8, prefix, div, extra=(3000, 17, 4100))
        _check_all(got, exp, vmax, "prefix %d" % prefix)
        assert counts[pkv.PKV_KERNEL_PREFILL] == 1


@pytest.mark.gpu
def test_cascade_needs_sixteen_rows(cascade_mode):
    div = [2] * 15
    got, exp, counts, vmax = _forks_then_decode(32, 8, 4096, div)
    _check_all(got, exp, vmax, "15 forks")
    assert counts[pkv.PKV_KERNEL_PREFILL] == 0
    assert counts["work"]["prefix_pairs"] == 0
