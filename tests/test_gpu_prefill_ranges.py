"""The tensor-core prefill kernel over inputs far from unit scale.

The kernel multiplies each query row, and each 64-key tile of K and of V
(per kv head), by a power of two before splitting it into two f16 pieces,
and scales the probabilities of a tile by 2^(C - c), where C is an exponent
that only decreases as tiles with larger V arrive (the accumulator is
rescaled exactly when it moves).  These cases drive those paths against the
oracle at the tests' tolerance (1e-5 max|V| + 1e-6): V tiles whose
magnitudes spread over 2^-30 .. 2^30 arriving in increasing order (C moves
on every tile; neighbouring tiles differ by 2^2.6, so a missed rescale
shows) and over 2^-8 .. 2^8 in random order per kv head; query rows and K tiles
spread over 2^-20 .. 2^2 (near-uniform rows beside sharp ones, lazy max
rescales); all-zero K and V tiles and query rows; and tiles whose largest
magnitudes sit far out in f32's range, subnormals included (the
exponents' clamps).  Each case also runs through a pool, which must return the
contiguous entry point's bits.  On bf16 / fp8 pools (the kernel's one-piece
K/V images) K and V tiles spread over 2^-6 .. 2^2 and 2^-8 .. 2^8 per kv
head, against the oracle over the rounded history.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool, assert_close, bits_equal, contiguous_attend

H, KV, HD = 32, 8, 128
TILE = 64


def _tiles(n):
    return [(t0, min(t0 + TILE, n)) for t0 in range(0, n, TILE)]


def _case(name, rng, n_q, total_k):
    Q = rng.standard_normal((n_q, H * HD)).astype(np.float32)
    K = rng.standard_normal((total_k, KV * HD)).astype(np.float32)
    V = rng.standard_normal((total_k, KV * HD)).astype(np.float32)
    tiles = _tiles(total_k)
    if name == "v_increasing":
        for i, (a, b) in enumerate(tiles):
            V[a:b] *= np.float32(2.0 ** (-30 + 60 * i / max(1, len(tiles) - 1)))
    elif name == "v_random_per_head":
        # 2^-8 .. 2^8 per (tile, kv head): C moves on many tiles while the
        # outputs stay comparable to max|V| (so the tolerance sees any slip)
        for a, b in tiles:
            for h in range(KV):
                V[a:b, h * HD:(h + 1) * HD] *= np.float32(2.0 ** rng.integers(-8, 9))
    elif name == "qk_ranges":
        # combined Q.K scale at most 2^3: the tolerance bounds a score's error
        # by about 1e-5 (base 2), which f32 arithmetic itself meets only while
        # sum_d |q_d k_d| (base 2) stays below about 100 (scaled up 2^6 instead,
        # one rounding per exact-f32 score already costs 1e-4 here)
        for r in range(n_q):
            for h in range(H):
                Q[r, h * HD:(h + 1) * HD] *= np.float32(2.0 ** rng.choice([-20, 0, 2]))
        for a, b in tiles:
            for h in range(KV):
                K[a:b, h * HD:(h + 1) * HD] *= np.float32(2.0 ** rng.integers(-20, 2))
    elif name == "zero_tiles":
        for i, (a, b) in enumerate(tiles):
            if i % 3 == 1:
                K[a:b] = 0.0
            if i % 4 == 2:
                V[a:b] = 0.0
        Q[::7] = 0.0
    elif name == "extremes":
        # largest magnitudes far out in f32's range: huge Q against tiny K
        # (scores of order one), V tiles from 1e-40 (subnormal) to 1e30 (the
        # sums p.v of a row, up to l = sum p times max|V|, stay finite in f32)
        Q *= np.float32(1e30)
        K *= np.float32(1e-31)
        for i, (a, b) in enumerate(tiles):
            V[a:b] *= np.float32([1e-40, 1e30, 1e-20, 1.0][i % 4])
    else:
        raise AssertionError(name)
    return Q, K, V


def _paged(Q, K, V, n_q, total_k, causal, scale):
    past = total_k - n_q
    kv_dim = KV * HD
    bs = 16
    blocks = -(-total_k // bs)
    pool = GpuPool(blocks + 4, 1, kv_dim, bs, max_seqs=2, max_blocks=blocks + 1, shuffle_seed=5)
    try:
        s = pool.new_seq(total_k)
        if past:
            pool.grow(s, past)
            pool.write_history(s, 0, torch.from_numpy(K[:past]), torch.from_numpy(V[:past]))
        pkv.check(pkv.pkv_ensure_append_batch([s], [n_q]))
        out = torch.empty(n_q, H * HD, device="cuda")
        Qd, Kd, Vd = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (Q, K[past:], V[past:]))
        pkv.check(pkv.pkv_attn_batch([s], [n_q], Qd, Kd, Vd, H, KV, HD, 0, causal, scale, out))
        pool.check_no_device_error()
        return out
    finally:
        pool.close()


@pytest.mark.gpu
@pytest.mark.parametrize("name,n_q,total_k,causal", [
    ("v_increasing", 96, 1500, 1),
    ("v_random_per_head", 64, 1300, 1),
    ("qk_ranges", 128, 1100, 1),
    ("zero_tiles", 70, 900, 1),
    ("extremes", 64, 1050, 0),
])
def test_prefill_far_from_unit_scale(name, n_q, total_k, causal):
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    Q, K, V = _case(name, rng, n_q, total_k)
    scale = float(np.float32(1.0 / math.sqrt(HD)))
    Qd, Kc, Vc = (torch.from_numpy(x).cuda() for x in (Q, K, V))
    out = contiguous_attend(Qd, Kc, Vc, n_q, total_k, H, KV, HD, causal, scale)
    assert pkv.pkv_contiguous_sync_error(torch.cuda.current_stream()) == pkv.PKV_OK, pkv.pkv_last_error()
    rc, exp = oracle.attend(Q, K, V, n_q, total_k, H, KV, HD, causal, scale)
    assert rc == 0
    assert_close(out.cpu().numpy(), exp, np.abs(V).max(), name)
    out_p = _paged(Q, K, V, n_q, total_k, causal, scale)
    assert bits_equal(out_p, out), name + ": paged != contiguous"


NARROW = {
    "bf16": (torch.bfloat16, 1.0, lambda x, s: oracle.round_bf16(x)),
    "fp8": (torch.float8_e4m3fn, 1.0, lambda x, s: oracle.round_e4m3(x, s)),
    "fp8s": (torch.float8_e4m3fn, 0.25, lambda x, s: oracle.round_e4m3(x, s)),
}


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["bf16", "fp8", "fp8s"])
def test_prefill_narrow_pool_ranges(fmt):
    """bf16 / fp8 pools take the kernel's one-piece K/V images (a pool value
    times its tile's power of two is an f16 value); here K tiles spread over
    2^-6 .. 2^2 and V tiles over 2^-8 .. 2^8 per kv head (on fp8 pools the
    largest saturate and the smallest fall into e4m3's subnormals, exactly as
    the oracle's rounding has them), against the oracle over the rounded
    history at the tests' tolerance."""
    dtype, kv_scale, rnd = NARROW[fmt]
    rng = np.random.default_rng(zlib.crc32(fmt.encode()) + 7)
    past, n_q, bs = 1000, 96, 16
    total_k = past + n_q
    kv_dim = KV * HD
    scale = float(np.float32(1.0 / math.sqrt(HD)))
    K = rng.standard_normal((total_k, kv_dim)).astype(np.float32)
    V = rng.standard_normal((total_k, kv_dim)).astype(np.float32)
    for a, b in _tiles(total_k):
        for h in range(KV):
            K[a:b, h * HD:(h + 1) * HD] *= np.float32(2.0 ** rng.integers(-6, 3))
            V[a:b, h * HD:(h + 1) * HD] *= np.float32(2.0 ** rng.integers(-8, 9))
    Q = rng.standard_normal((n_q, H * HD)).astype(np.float32)
    # the oracle's rounding (saturating at +-448 x scale on fp8 pools, as the
    # library's store does); the history is written as those exact values,
    # since torch's e4m3fn cast turns magnitudes beyond 448 into NaN
    Kr, Vr = rnd(K, kv_scale), rnd(V, kv_scale)
    blocks = -(-total_k // bs)
    pool = GpuPool(blocks + 4, 1, kv_dim, bs, max_seqs=2, max_blocks=blocks + 1, shuffle_seed=3,
                   dtype=dtype, kv_scale=kv_scale)
    try:
        s = pool.new_seq(total_k)
        pool.grow(s, past)
        pool.write_history(s, 0, torch.from_numpy(Kr[:past]), torch.from_numpy(Vr[:past]))
        pkv.check(pkv.pkv_ensure_append_batch([s], [n_q]))
        out = torch.empty(n_q, H * HD, device="cuda")
        Qd, Kd, Vd = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (Q, K[past:], V[past:]))
        pkv.check(pkv.pkv_attn_batch([s], [n_q], Qd, Kd, Vd, H, KV, HD, 0, 1, scale, out))
        pool.check_no_device_error()
        rc, exp = oracle.attend(Q, Kr, Vr, n_q, total_k, H, KV, HD, 1, scale)
        assert rc == 0
        assert_close(out.cpu().numpy(), exp, np.abs(Vr).max(), fmt)
    finally:
        pool.close()
