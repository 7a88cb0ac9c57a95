"""Parity at the full workload sizes, through the same entry point and launch
configuration the benchmark times (pkv_attn_batch, default split size).

* batched decode, M = 64, Qwen3-4B attention shape: every row vs the oracle.
* continuous-batching decode, M = 256, log-uniform lengths, 600 000-block
  shuffled pool: every row vs the oracle, and the contiguous twin bit for
  bit on the shortest and the longest; the same step on bf16 and fp8 pools
  (the benchmark's --kv-dtype runs) vs the oracle over the rounded
  histories, on every row as well.
* chunked prefill, 8 x (2048 + 512) over 4 layers: every query of every row
  on the first and the last layer (all 16 query tiles of each row).
* shared-prefix forks: 128 forks of an 8192-token prefix, divergent chunks,
  a batched decode step, truncation of half the forks and re-append; and the
  same with an unaligned 8200-token prefix, where copy-on-append fires.

Histories are drawn with seeded torch generators and written into the pool
with torch indexing; the oracle receives host copies of those draws (drawn
again from the same seeds when a row is checked, so that the whole M = 256
history never sits in host memory at once).  The oracle runs on every host
core; its result does not depend on the thread count.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from synth import workloads as wl
from gpu_helpers import GpuPool, assert_close, bits_equal, contiguous_attend


def _oracle_row(Qr, Kf, Vf, n, tk, w, causal=1):
    rc, ref = oracle.attend(Qr, Kf, Vf, n, tk, w.n_heads, w.n_kv_heads, w.head_dim, causal, w.scale)
    assert rc == 0
    return ref


# pool element -> (torch dtype, the oracle's rounding of the values a row reads back)
FORMATS = {
    "f32": (torch.float32, lambda x: x),
    "bf16": (torch.bfloat16, oracle.round_bf16),
    "fp8": (torch.float8_e4m3fn, lambda x: oracle.round_e4m3(x, 1.0)),
}


def _history(w, r, seed_base):
    """Row r's K and V history draws (device), as build_decode writes them."""
    L = int(w.past_len[r])
    return (wl.normal((L, w.kv_dim), seed_base + 2 * r, "cuda"),
            wl.normal((L, w.kv_dim), seed_base + 2 * r + 1, "cuda"))


def build_decode(w, seed_base, fmt="f32"):
    """Pool + sequences holding each row's history (layer 0)."""
    dtype, _ = FORMATS[fmt]
    pool = GpuPool(w.n_blocks, w.n_layers, w.kv_dim, w.block_size, max_seqs=w.M + 4,
                   max_blocks=-(-(w.max_tokens() + 1) // w.block_size) + 1, shuffle_seed=w.seed,
                   dtype=dtype)
    seqs = []
    for r in range(w.M):
        L = int(w.past_len[r])
        s = pool.new_seq(L + int(w.n_q[r]) + 1)
        pool.grow(s, L)
        Kh, Vh = _history(w, r, seed_base)
        pool.write_history(s, 0, Kh, Vh)
        del Kh, Vh
        seqs.append(s)
    torch.cuda.synchronize()
    return pool, seqs


def decode_step_and_check(w, rows_to_check, contig_rows=(), fmt="f32"):
    rnd = FORMATS[fmt][1]
    seed_base = w.seed * 1000
    pool, seqs = build_decode(w, seed_base, fmt)
    try:
        T = int(w.n_q.sum())
        Q = wl.normal((T, w.q_dim), w.seed + 101, "cuda")
        Kn = wl.normal((T, w.kv_dim), w.seed + 102, "cuda")
        Vn = wl.normal((T, w.kv_dim), w.seed + 103, "cuda")
        nq = [int(x) for x in w.n_q]
        pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
        out = torch.empty(T, w.q_dim, device="cuda")
        pkv.check(pkv.pkv_attn_batch(seqs, nq, Q, Kn, Vn, w.n_heads, w.n_kv_heads, w.head_dim, 0, 1,
                                     w.scale, out))
        pool.check_no_device_error()
        offs = np.concatenate([[0], np.cumsum(w.n_q)])
        Qh, Knh, Vnh, outh = Q.cpu().numpy(), Kn.cpu().numpy(), Vn.cpu().numpy(), out.cpu().numpy()
        for r in rows_to_check:
            o, n, L = int(offs[r]), nq[r], int(w.past_len[r])
            Kd, Vd = _history(w, r, seed_base)
            Kf = np.concatenate([rnd(Kd.cpu().numpy()), rnd(Knh[o:o + n])])
            Vf = np.concatenate([rnd(Vd.cpu().numpy()), rnd(Vnh[o:o + n])])
            del Kd, Vd
            ref = _oracle_row(Qh[o:o + n], Kf, Vf, n, L + n, w)
            assert_close(outh[o:o + n], ref, np.abs(Vf).max(), "%s row %d (len %d)" % (w.name, r, L))
            if r in contig_rows:
                oc = contiguous_attend(Q[o:o + n], torch.from_numpy(Kf).cuda(), torch.from_numpy(Vf).cuda(),
                                       n, L + n, w.n_heads, w.n_kv_heads, w.head_dim, 1, w.scale)
                assert bits_equal(out[o:o + n], oc)
    finally:
        pool.close()


@pytest.mark.gpu
def test_batched_decode_m64_all_rows():
    w = wl.batched_decode_m64()
    decode_step_and_check(w, list(range(w.M)), contig_rows=(0, 1))


@pytest.mark.gpu
def test_continuous_batching_m256_all_rows():
    w = wl.continuous_batching_m256()
    free, _ = torch.cuda.mem_get_info()
    need = 2 * w.n_blocks * w.block_size * w.kv_dim * 4
    if free < need + (8 << 30):
        pytest.skip("needs %.1f GB of device memory" % (need / 1e9))
    decode_step_and_check(w, list(range(w.M)),
                          contig_rows=(int(np.argmin(w.past_len)), int(np.argmax(w.past_len))))


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
def test_continuous_batching_m256_narrow_pool_all_rows(fmt):
    w = wl.continuous_batching_m256()
    free, _ = torch.cuda.mem_get_info()
    need = 2 * w.n_blocks * w.block_size * w.kv_dim * (2 if fmt == "bf16" else 1)
    if free < need + (8 << 30):
        pytest.skip("needs %.1f GB of device memory" % (need / 1e9))
    decode_step_and_check(w, list(range(w.M)), fmt=fmt)


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["f32", "bf16"])
def test_chunked_prefill_every_query(fmt):
    w = wl.chunked_prefill()
    bs = w.block_size
    dtype, rnd = FORMATS[fmt]
    pool = GpuPool(w.n_blocks, w.n_layers, w.kv_dim, bs, max_seqs=w.M + 2,
                   max_blocks=-(-w.max_tokens() // bs) + 1, shuffle_seed=w.seed, dtype=dtype)
    try:
        past, n = int(w.past_len[0]), int(w.n_q[0])
        seqs, hist = [], {}
        for r in range(w.M):
            s = pool.new_seq(past + n)
            pool.grow(s, past)
            for layer in range(w.n_layers):
                Kh = wl.normal((past, w.kv_dim), w.seed * 100 + 10 * r + 2 * layer, "cuda")
                Vh = wl.normal((past, w.kv_dim), w.seed * 100 + 10 * r + 2 * layer + 1, "cuda")
                pool.write_history(s, layer, Kh, Vh)
                if layer in (0, w.n_layers - 1):
                    hist[(r, layer)] = (rnd(Kh.cpu().numpy()), rnd(Vh.cpu().numpy()))
            seqs.append(s)
        T = w.M * n
        nq = [n] * w.M
        pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
        results = []
        for layer in range(w.n_layers):
            Q = wl.normal((T, w.q_dim), w.seed + 200 + layer, "cuda")
            Kn = wl.normal((T, w.kv_dim), w.seed + 300 + layer, "cuda")
            Vn = wl.normal((T, w.kv_dim), w.seed + 400 + layer, "cuda")
            out = torch.empty(T, w.q_dim, device="cuda")
            pkv.check(pkv.pkv_attn_batch(seqs, nq, Q, Kn, Vn, w.n_heads, w.n_kv_heads, w.head_dim,
                                         layer, 1, w.scale, out))
            results.append((Q.cpu().numpy(), Kn.cpu().numpy(), Vn.cpu().numpy(), out.cpu().numpy()))
        pkv.check(pkv.pkv_advance_batch(seqs, nq))
        pool.check_no_device_error()
        for layer in (0, w.n_layers - 1):
            Qh, Knh, Vnh, outh = results[layer]
            for r in range(w.M):
                Kf = np.concatenate([hist[(r, layer)][0], rnd(Knh[r * n:(r + 1) * n])])
                Vf = np.concatenate([hist[(r, layer)][1], rnd(Vnh[r * n:(r + 1) * n])])
                # all n queries of the row at once: query i sits at past + i
                ref = _oracle_row(Qh[r * n:(r + 1) * n], Kf, Vf, n, past + n, w)
                got = outh[r * n:(r + 1) * n]
                vmax = np.abs(Vf).max()
                for t0 in range(0, n, 32):  # report the failing 32-query tile, if any
                    assert_close(got[t0:t0 + 32], ref[t0:t0 + 32], vmax,
                                 "layer %d row %d queries %d..%d" % (layer, r, t0, t0 + 31))
    finally:
        pool.close()


def _shared_prefix(prefix, n_forks, seed):
    w = wl.shared_prefix_forks(prefix=prefix, n_forks=n_forks)
    bs = w.block_size
    div = [int(x) for x in w.n_q]
    pool = GpuPool(w.n_blocks, 1, w.kv_dim, bs, max_seqs=n_forks + 4,
                   max_blocks=-(-(prefix + 2 * 256 + 2) // bs) + 1, shuffle_seed=w.seed)
    try:
        root = pool.new_seq(prefix + 2 * 256 + 2)
        pool.grow(root, prefix)
        Kp = wl.normal((prefix, w.kv_dim), seed, "cuda")
        Vp = wl.normal((prefix, w.kv_dim), seed + 1, "cuda")
        pool.write_history(root, 0, Kp, Vp)
        Kp_h, Vp_h = Kp.cpu().numpy(), Vp.cpu().numpy()
        forks = [pkv.pkv_seq_fork(root) for _ in range(n_forks)]
        assert all(forks)
        pt_root = pkv.pkv_seq_page_table(root)
        assert pkv.pkv_refcnt(pool.p, pt_root[0]) == n_forks + 1
        check = sorted({0, n_forks // 2, n_forks - 1, int(np.argmax(div))})

        def chunk_round(seqs, ns, tag, hist):
            T = sum(ns)
            Q = wl.normal((T, w.q_dim), seed + tag, "cuda")
            K = wl.normal((T, w.kv_dim), seed + tag + 1, "cuda")
            V = wl.normal((T, w.kv_dim), seed + tag + 2, "cuda")
            pkv.check(pkv.pkv_ensure_append_batch(seqs, ns))
            out = torch.empty(T, w.q_dim, device="cuda")
            pkv.check(pkv.pkv_attn_batch(seqs, ns, Q, K, V, w.n_heads, w.n_kv_heads, w.head_dim, 0, 1,
                                         w.scale, out))
            pkv.check(pkv.pkv_advance_batch(seqs, ns))
            Qh, Kh, Vh, oh = Q.cpu().numpy(), K.cpu().numpy(), V.cpu().numpy(), out.cpu().numpy()
            o = 0
            for j, (s, n) in enumerate(zip(seqs, ns)):
                kh, vh = hist[s]
                hist[s] = (np.concatenate([kh, Kh[o:o + n]]), np.concatenate([vh, Vh[o:o + n]]))
                if j in check:
                    Kf, Vf = hist[s]
                    ref = _oracle_row(Qh[o:o + n], Kf, Vf, n, Kf.shape[0], w)
                    assert_close(oh[o:o + n], ref, np.abs(Vf).max(), "fork %d tag %d" % (j, tag))
                o += n

        hist = {f: (Kp_h, Vp_h) for f in forks}
        chunk_round(forks, div, 10, hist)                      # divergent chunks (copy-on-append)
        for f in forks:
            pt = pkv.pkv_seq_page_table(f)
            assert pt[:prefix // bs] == pt_root[:prefix // bs]  # full prefix blocks stay shared
        chunk_round(forks, [1] * n_forks, 20, hist)             # batched decode step of all forks
        half = forks[: n_forks // 2]
        for f in half:
            pkv.check(pkv.pkv_seq_truncate(f, prefix))
            hist[f] = (Kp_h, Vp_h)
        chunk_round(half, div[: n_forks // 2], 30, hist)        # re-append fresh divergent chunks
        assert pkv.pkv_seq_len(root) == prefix
        pool.check_no_device_error()
    finally:
        pool.close()


@pytest.mark.gpu
def test_shared_prefix_forks_aligned():
    _shared_prefix(8192, 128, 77)


@pytest.mark.gpu
def test_shared_prefix_forks_unaligned_cow():
    _shared_prefix(8200, 16, 88)
