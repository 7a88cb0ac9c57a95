"""RoPE on append against the oracle.

"nx_f32_llama_v4b.nx source", Block section: the queries and the new keys of
each row are rotated (NeoX pairing) at the row's position, its sequence's
length, before the attend call; V is not rotated.  The oracle rotates the same
generator draws in float64 and attends over [history; rotated new keys]; the
histories in the pool stand for keys appended (and rotated) earlier and are
used as they are.  Also checked: the rotated key rows that land in the pool,
that the caller's Q and K_new are untouched, and the argument checks.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool, assert_close, bits_equal


def _rope_case(H, KV, hd, past, nq, base, seed=0, bs=16):
    rng = np.random.default_rng(seed)
    kv_dim, q_dim = KV * hd, H * hd
    scale = float(np.float32(1.0 / math.sqrt(hd)))
    need = sum(-(-(p + n) // bs) for p, n in zip(past, nq))
    pool = GpuPool(need + 8, 1, kv_dim, bs, max_seqs=len(past) + 2,
                   max_blocks=max(-(-(p + n) // bs) for p, n in zip(past, nq)) + 1, shuffle_seed=seed + 3)
    try:
        seqs, hk, hv = [], [], []
        for p, n in zip(past, nq):
            s = pool.new_seq(p + n)
            Kh = rng.standard_normal((p, kv_dim)).astype(np.float32)
            Vh = rng.standard_normal((p, kv_dim)).astype(np.float32)
            if p:
                pool.grow(s, p)
                pool.write_history(s, 0, torch.from_numpy(Kh), torch.from_numpy(Vh))
            seqs.append(s)
            hk.append(Kh)
            hv.append(Vh)
        T = int(sum(nq))
        Q = rng.standard_normal((T, q_dim)).astype(np.float32)
        Kn = rng.standard_normal((T, kv_dim)).astype(np.float32)
        Vn = rng.standard_normal((T, kv_dim)).astype(np.float32)
        Qd, Kd, Vd = (torch.from_numpy(a).cuda() for a in (Q, Kn, Vn))
        Q0, K0 = Qd.clone(), Kd.clone()
        pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
        out = torch.empty(T, q_dim, device="cuda")
        pkv.check(pkv.pkv_attn_batch_rope(seqs, nq, Qd, Kd, Vd, H, KV, hd, 0, 1, scale, base, out))
        pool.check_no_device_error()
        assert bits_equal(Qd, Q0) and bits_equal(Kd, K0), "caller's Q / K_new changed"
        got = out.cpu().numpy()
        o = 0
        for r, (p, n) in enumerate(zip(past, nq)):
            pos = np.arange(p, p + n)
            Qr = oracle.rope_neox(Q[o:o + n], pos, hd, base)
            Kr = oracle.rope_neox(Kn[o:o + n], pos, hd, base)
            # the rotated new keys in the pool (f32 rotation vs the float64 one)
            Kpool, _ = pool.read_history(seqs[r], 0, p + n)
            kp = Kpool[p:].cpu().numpy().astype(np.float64)
            assert np.max(np.abs(kp - Kr)) <= 4e-7 * max(1.0, np.abs(Kr).max()), "row %d: pool keys" % r
            Kf = np.concatenate([hk[r], Kr]).astype(np.float32)
            Vf = np.concatenate([hv[r], Vn[o:o + n]])
            rc, ref = oracle.attend(Qr.astype(np.float32), Kf, Vf, n, p + n, H, KV, hd, 1, scale)
            assert rc == 0
            assert_close(got[o:o + n], ref, np.abs(Vf).max(), "row %d" % r)
            o += n
    finally:
        pool.close()


@pytest.mark.gpu
@pytest.mark.parametrize("base", [10000.0, 1000000.0], ids=["base1e4", "base1e6"])
def test_rope_fast_kernel_rows(base):
    # decode rows, a multi-token row and a tensor-core prefill row; positions up to 30k
    _rope_case(32, 8, 128, [0, 5, 1000, 30000, 2100], [1, 3, 1, 1, 64], base)


@pytest.mark.gpu
def test_rope_generic_kernel_odd_pairs():
    # head_dim 10: pairs (i, i + 5); the generic decode kernel
    _rope_case(4, 2, 10, [0, 17, 300], [1, 2, 5], 10000.0, seed=1, bs=4)


@pytest.mark.gpu
def test_rope_argument_checks_change_nothing():
    pool = GpuPool(8, 1, 5, 4, max_seqs=2, max_blocks=4)
    try:
        s = pool.new_seq(8)
        pkv.check(pkv.pkv_ensure_append(s, 1))
        Q = torch.zeros(1, 10, device="cuda")
        K = torch.zeros(1, 5, device="cuda")
        out = torch.empty(1, 10, device="cuda")
        # odd head_dim
        assert pkv.pkv_attn_batch_rope([s], [1], Q, K, K, 2, 1, 5, 0, 1, 1.0, 10000.0, out) == pkv.PKV_ERR_BAD_DIM
        pool2 = GpuPool(8, 1, 4, 4, max_seqs=2, max_blocks=4)
        try:
            s2 = pool2.new_seq(8)
            pkv.check(pkv.pkv_ensure_append(s2, 1))
            Q2 = torch.zeros(1, 8, device="cuda")
            K2 = torch.zeros(1, 4, device="cuda")
            out2 = torch.empty(1, 8, device="cuda")
            for bad in (0.0, -3.0):
                assert pkv.pkv_attn_batch_rope([s2], [1], Q2, K2, K2, 2, 1, 4, 0, 1, 1.0, bad, out2) == pkv.PKV_ERR_ARG
            assert pkv.pkv_seq_len(s2) == 0
        finally:
            pool2.close()
        assert pkv.pkv_seq_len(s) == 0
    finally:
        pool.close()
