"""bf16 and fp8 K/V pools (PKV_POOL_BF16 / PKV_POOL_FP8; not on the pages,
which store f32).

Every K/V row is rounded once when it is written -- to the nearest bfloat16,
or to e4m3 of x / scale (saturating, scale a power of two) -- and read back
exactly; the attention math stays f32.  So the oracle attends, in its usual
precision, over the rounded histories: the rows written into the pool with
torch's casts (which the oracle's round_bf16 / round_e4m3 match, pinned on
the CPU) and the call's new rows rounded by the oracle.  The values the
library stores are compared with the oracle's rounding bit for bit.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool, assert_close, bits_equal

BF = torch.bfloat16
FMTS = {
    "bf16": (torch.bfloat16, 1.0, lambda x, s: oracle.round_bf16(x)),
    "fp8": (torch.float8_e4m3fn, 1.0, lambda x, s: oracle.round_e4m3(x, s)),
    "fp8s": (torch.float8_e4m3fn, 0.25, lambda x, s: oracle.round_e4m3(x, s)),
}


def _case(H, KV, hd, past, nq, seed=0, bs=16, rope=0.0, check_m1=True, fmt="bf16", q_head_scale=None):
    dtype, kv_scale, rnd = FMTS[fmt]
    rng = np.random.default_rng(seed)
    kv_dim, q_dim = KV * hd, H * hd
    scale = float(np.float32(1.0 / math.sqrt(hd)))
    need = sum(-(-(p + n) // bs) for p, n in zip(past, nq))
    pool = GpuPool(need + 8, 1, kv_dim, bs, max_seqs=len(past) + 2,
                   max_blocks=max(-(-(p + n) // bs) for p, n in zip(past, nq)) + 1,
                   shuffle_seed=seed + 5, dtype=dtype, kv_scale=kv_scale)
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
            hk.append(rnd(Kh, kv_scale))
            hv.append(rnd(Vh, kv_scale))
        T = int(sum(nq))
        Q = rng.standard_normal((T, q_dim)).astype(np.float32)
        if q_head_scale is not None:  # per query head magnitudes
            Q = (Q.reshape(T, H, hd) * np.asarray(q_head_scale, np.float32)[None, :, None]).reshape(T, q_dim)
        Kn = rng.standard_normal((T, kv_dim)).astype(np.float32)
        Vn = rng.standard_normal((T, kv_dim)).astype(np.float32)
        Qd, Kd, Vd = (torch.from_numpy(a).cuda() for a in (Q, Kn, Vn))
        pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
        out = torch.empty(T, q_dim, device="cuda")
        if rope:
            pkv.check(pkv.pkv_attn_batch_rope(seqs, nq, Qd, Kd, Vd, H, KV, hd, 0, 1, scale, rope, out))
        else:
            pkv.check(pkv.pkv_attn_batch(seqs, nq, Qd, Kd, Vd, H, KV, hd, 0, 1, scale, out))
        pool.check_no_device_error()
        got = out.cpu().numpy()
        o = 0
        for r, (p, n) in enumerate(zip(past, nq)):
            pos = np.arange(p, p + n)
            Qr, Kr = Q[o:o + n], Kn[o:o + n]
            if rope:
                # the rotated keys are rounded to bf16: the oracle takes that
                # rounding decision on the same float32 values the kernel rounds
                Qr = oracle.rope_neox(Qr, pos, hd, rope).astype(np.float32)
                Kr = oracle.rope_neox_f32(Kr, pos, hd, rope)
            Kr, Vr = rnd(Kr, kv_scale), rnd(Vn[o:o + n], kv_scale)
            Kp, Vp = pool.read_values(seqs[r], 0, p + n)
            stored_k = Kp[p:].cpu().numpy()
            stored_v = Vp[p:].cpu().numpy()
            assert np.array_equal(stored_k.view(np.uint32), Kr.view(np.uint32)), "row %d K" % r
            assert np.array_equal(stored_v.view(np.uint32), Vr.view(np.uint32)), "row %d V" % r
            Kf = np.concatenate([hk[r], Kr])
            Vf = np.concatenate([hv[r], Vr])
            rc, ref = oracle.attend(Qr, Kf, Vf, n, p + n, H, KV, hd, 1, scale)
            assert rc == 0
            assert_close(got[o:o + n], ref, np.abs(Vf).max(), "row %d" % r)
            if check_m1 and not rope:
                o1 = torch.empty(n, q_dim, device="cuda")
                pkv.check(pkv.pkv_attn_with_paged(Qd[o:o + n], Kd[o:o + n], Vd[o:o + n], n, H, KV, hd,
                                                  seqs[r], 0, 1, scale, o1))
                assert bits_equal(out[o:o + n], o1), "row %d: batched != M=1" % r
            o += n
        pool.check_no_device_error()
    finally:
        pool.close()


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["bf16", "fp8", "fp8s"])
@pytest.mark.parametrize("H,KV", [(32, 8), (16, 8), (8, 8)], ids=["g4", "g2", "g1"])
def test_narrow_decode_and_prefill(H, KV, fmt):
    # decode rows across page and split boundaries, a short multi-token row, a
    # tensor-core prefill row
    _case(H, KV, 128, [0, 15, 1024, 3000, 777, 2100], [1, 1, 1, 1, 5, 64], fmt=fmt)


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["fp8", "fp8s"])
def test_fp8_group8(fmt):
    # 64 query heads on 8 kv heads: the fp8 tensor-core kernel carries all 8
    # heads of a group in one MMA tile
    _case(64, 8, 128, [0, 31, 1024, 2500, 100], [1, 1, 1, 1, 7], seed=4, fmt=fmt)


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
def test_narrow_small_pages(fmt):
    # 8-row pages: every key of a tile is looked up on its own
    _case(32, 8, 128, [0, 13, 1030, 333], [1, 1, 3, 1], seed=5, bs=8, fmt=fmt)


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["bf16", "fp8", "fp8s"])
def test_narrow_query_magnitudes(fmt):
    # query heads from 1e-4 to 8 in size (scores from nearly uniform to
    # sharply peaked; larger scores would put the f32 rounding of the scores
    # themselves above the tolerance); the f16 pieces of an fp8 pool are
    # scaled per head
    H = 32
    sc = [1e-4 * (8e4 ** (i / (H - 1))) for i in range(H)]
    _case(H, 8, 128, [5, 700, 2049], [1, 1, 2], seed=6, fmt=fmt, q_head_scale=sc)


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["bf16", "fp8s"])
def test_narrow_generic_kernel(fmt):
    # head_dim 8 (generic kernel), 4-row pages
    _case(6, 2, 8, [0, 9, 130], [1, 3, 1], seed=2, bs=4, fmt=fmt)


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
def test_narrow_rope_on_append(fmt):
    _case(32, 8, 128, [0, 100, 5000], [1, 2, 40], seed=3, rope=10000.0, fmt=fmt)


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["bf16", "fp8s"])
def test_narrow_copy_on_append_and_cascade(fmt):
    # forks of a narrow-pool prefix ending inside a page: the first append
    # copies the tail page (2- or 1-byte elements); then a batched decode step
    # of 20 forks takes the shared-prefix path.  Every fork is checked against
    # the oracle.
    dtype, kv_scale, rnd0 = FMTS[fmt]
    rnd = lambda x: rnd0(x, kv_scale)  # noqa: E731
    H, KV, hd, bs = 32, 8, 128, 16
    kv_dim, q_dim = KV * hd, H * hd
    scale = float(np.float32(1.0 / math.sqrt(hd)))
    rng = np.random.default_rng(9)
    prefix, n_f = 2500, 20
    pool = GpuPool(prefix // bs + 4 * n_f + 16, 1, kv_dim, bs, max_seqs=n_f + 4,
                   max_blocks=prefix // bs + 8, shuffle_seed=4, dtype=dtype, kv_scale=kv_scale)
    try:
        root = pool.new_seq(prefix + 40)
        Kp = rng.standard_normal((prefix, kv_dim)).astype(np.float32)
        Vp = rng.standard_normal((prefix, kv_dim)).astype(np.float32)
        pool.grow(root, prefix)
        pool.write_history(root, 0, torch.from_numpy(Kp), torch.from_numpy(Vp))
        forks = [pkv.pkv_seq_fork(root) for _ in range(n_f)]
        hist = {f: (rnd(Kp), rnd(Vp)) for f in forks}
        for tag, n in ((1, 3), (2, 1)):
            M = len(forks)
            Q = rng.standard_normal((M * n, q_dim)).astype(np.float32)
            Kn = rng.standard_normal((M * n, kv_dim)).astype(np.float32)
            Vn = rng.standard_normal((M * n, kv_dim)).astype(np.float32)
            pkv.check(pkv.pkv_ensure_append_batch(forks, [n] * M))
            out = torch.empty(M * n, q_dim, device="cuda")
            pkv.pkv_profile_reset()
            pkv.pkv_profile_enable(True)
            pkv.check(pkv.pkv_attn_batch(forks, [n] * M, torch.from_numpy(Q).cuda(),
                                         torch.from_numpy(Kn).cuda(), torch.from_numpy(Vn).cuda(),
                                         H, KV, hd, 0, 1, scale, out))
            torch.cuda.synchronize()
            pkv.pkv_profile_enable(False)
            n_pre = pkv.pkv_profile_read(pkv.PKV_KERNEL_PREFILL)[1]
            pkv.pkv_profile_reset()
            pkv.check(pkv.pkv_advance_batch(forks, [n] * M))
            pool.check_no_device_error()
            got = out.cpu().numpy()
            for j, f in enumerate(forks):
                kh, vh = hist[f]
                kh = np.concatenate([kh, rnd(Kn[j * n:(j + 1) * n])])
                vh = np.concatenate([vh, rnd(Vn[j * n:(j + 1) * n])])
                hist[f] = (kh, vh)
                rc, ref = oracle.attend(Q[j * n:(j + 1) * n], kh, vh, n, kh.shape[0], H, KV, hd, 1, scale)
                assert rc == 0
                assert_close(got[j * n:(j + 1) * n], ref, np.abs(vh).max(), "tag %d fork %d" % (tag, j))
            if tag == 2:
                assert n_pre == 1, "the decode step should take the shared-prefix pass"
        # the root still sees its own prefix, untouched by the forks' copies
        Kr, _ = pool.read_values(root, 0, prefix)
        assert np.array_equal(Kr.cpu().numpy().view(np.uint32), rnd(Kp).view(np.uint32))
    finally:
        pool.close()


@pytest.mark.gpu
def test_narrow_pool_argument_checks():
    K = torch.zeros(4, 1, 4, 5, device="cuda", dtype=BF)
    assert not pkv.pkv_pool_new(4, 1, 5, 4, K, K.clone(), 2, 4, None, pkv.PKV_POOL_BF16)
    assert "even kv_dim" in pkv.pkv_last_error()
    K8 = torch.zeros(4, 1, 4, 6, device="cuda", dtype=torch.float8_e4m3fn)
    assert not pkv.pkv_pool_new(4, 1, 6, 4, K8, K8.clone(), 2, 4, None, pkv.PKV_POOL_FP8)
    assert "multiple of 4" in pkv.pkv_last_error()
    K8 = torch.zeros(4, 1, 4, 8, device="cuda", dtype=torch.float8_e4m3fn)
    p = pkv.pkv_pool_new(4, 1, 8, 4, K8, K8.clone(), 2, 4, None, pkv.PKV_POOL_FP8)
    assert p
    try:
        for bad in (3.0, 0.0, -2.0, 2.0 ** 30):
            assert pkv.pkv_pool_set_kv_scale(p, bad) == pkv.PKV_ERR_ARG
        assert pkv.pkv_pool_set_kv_scale(p, 0.5) == pkv.PKV_OK
        assert pkv.pkv_alloc_block(p) == 0
        assert pkv.pkv_pool_set_kv_scale(p, 2.0) == pkv.PKV_ERR_ARG  # a block is in use
    finally:
        pkv.pkv_pool_free(p)
