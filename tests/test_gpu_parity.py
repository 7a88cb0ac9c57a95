"""GPU parity on seeded shapes that span several tiles and splits with ragged
tails: the batched paged path against the oracle (within tolerance), against
the contiguous twin (bit for bit), against the same row launched alone (bit
for bit), and under a permutation of the physical blocks (bit for bit).

Shapes cover the head_dim-128 fast kernel (query groups 1, 2, 4) and the
generic kernel (head_dim 5..256, groups 1..32, block sizes 1..16 including
non-powers of two), decode rows (n_q = 1), chunked-prefill rows (n_q > 1,
offset-causal), non-causal rows, a first token (total_k = 1) and rows whose
length sits on and next to block and split boundaries.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool, assert_close, bits_equal, contiguous_attend


@pytest.fixture
def split_keys():
    old = pkv.pkv_get_split_keys()
    yield lambda k: pkv.check(pkv.pkv_set_split_keys(k))
    pkv.check(pkv.pkv_set_split_keys(old))


def run_case(H, KV, hd, bs, past, nq, causal=1, seed=0, n_layers=1, layer=0, shuffle=True,
             check_m1=True, check_contig=True, shape_data=None):
    rng = np.random.default_rng(seed)
    M = len(past)
    kv_dim, q_dim = KV * hd, H * hd
    scale = float(np.float32(1.0 / math.sqrt(hd)))
    need = sum(-(-(p + n) // bs) for p, n in zip(past, nq))
    max_blocks = max(-(-(p + n) // bs) for p, n in zip(past, nq)) + 1
    pool = GpuPool(need + 8, n_layers, kv_dim, bs, max_seqs=M + 2, max_blocks=max_blocks,
                   shuffle_seed=(seed + 11) if shuffle else None)
    try:
        seqs, hk, hv = [], [], []
        for p, n in zip(past, nq):
            s = pool.new_seq(p + n)
            Kh = rng.standard_normal((p, kv_dim)).astype(np.float32)
            Vh = rng.standard_normal((p, kv_dim)).astype(np.float32)
            if shape_data is not None:
                Kh = shape_data("K", Kh, 0)
            if p:
                pool.grow(s, p)
                pool.write_history(s, layer, torch.from_numpy(Kh), torch.from_numpy(Vh))
            seqs.append(s)
            hk.append(Kh)
            hv.append(Vh)
        T = int(sum(nq))
        Q = rng.standard_normal((T, q_dim)).astype(np.float32)
        Kn = rng.standard_normal((T, kv_dim)).astype(np.float32)
        Vn = rng.standard_normal((T, kv_dim)).astype(np.float32)
        if shape_data is not None:
            Q = shape_data("Q", Q, 0)
            o = 0
            for p, n in zip(past, nq):
                Kn[o:o + n] = shape_data("K", Kn[o:o + n], p)
                o += n
        Qd, Kd, Vd = (torch.from_numpy(a).cuda() for a in (Q, Kn, Vn))
        pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
        out = torch.empty(T, q_dim, device="cuda")
        pkv.check(pkv.pkv_attn_batch(seqs, nq, Qd, Kd, Vd, H, KV, hd, layer, causal, scale, out))
        pool.check_no_device_error()
        o = 0
        for r, (p, n) in enumerate(zip(past, nq)):
            Kf = np.concatenate([hk[r], Kn[o:o + n]])
            Vf = np.concatenate([hv[r], Vn[o:o + n]])
            rc, ref = oracle.attend(Q[o:o + n], Kf, Vf, n, p + n, H, KV, hd, causal, scale)
            assert rc == 0
            assert_close(out[o:o + n].cpu().numpy(), ref, np.abs(Vf).max(), "row %d" % r)
            if check_contig:
                oc = contiguous_attend(Qd[o:o + n], torch.from_numpy(Kf).cuda(),
                                       torch.from_numpy(Vf).cuda(), n, p + n, H, KV, hd, causal,
                                       scale)
                assert bits_equal(out[o:o + n], oc), "row %d: paged != contiguous" % r
            if check_m1:
                # the same row alone (re-appending the same rows at the same positions)
                o1 = torch.empty(n, q_dim, device="cuda")
                pkv.check(pkv.pkv_attn_with_paged(Qd[o:o + n], Kd[o:o + n], Vd[o:o + n], n, H, KV,
                                                  hd, seqs[r], layer, causal, scale, o1))
                assert bits_equal(out[o:o + n], o1), "row %d: batched != M=1" % r
            o += n
        pool.check_no_device_error()
        return out
    finally:
        pool.close()


EDGE_LENS = [0, 1, 7, 8, 15, 16, 17, 63, 64, 65, 511, 512, 513, 1000]


@pytest.mark.gpu
@pytest.mark.parametrize("H,KV", [(32, 8), (16, 8), (8, 8)], ids=["g4", "g2", "g1"])
def test_fast_kernel_decode(H, KV, split_keys):
    split_keys(512)
    run_case(H, KV, 128, 16, EDGE_LENS, [1] * len(EDGE_LENS), seed=H)


@pytest.mark.gpu
@pytest.mark.parametrize("split", [32, 64, 96])
def test_fast_kernel_many_splits(split, split_keys):
    split_keys(split)
    run_case(32, 8, 128, 16, [31, 32, 33, 200, 777, 1300], [1] * 6, seed=split)


@pytest.mark.gpu
def test_fast_kernel_prefill_rows(split_keys):
    split_keys(64)
    run_case(32, 8, 128, 16, [0, 5, 100, 64, 300], [1, 3, 17, 40, 70], seed=7)


@pytest.mark.gpu
def test_fast_kernel_noncausal(split_keys):
    split_keys(64)
    run_case(32, 8, 128, 16, [10, 90], [5, 33], causal=0, seed=8)


@pytest.mark.gpu
@pytest.mark.parametrize("H,KV,hd,bs", [
    (4, 2, 8, 4),        # the gate's shape
    (12, 3, 64, 5),      # non-power-of-two block size
    (32, 1, 64, 16),     # group 32 -> two head chunks
    (8, 2, 256, 16),     # largest head_dim
    (6, 2, 96, 3),
    (3, 1, 5, 4),        # kv_dim not a multiple of 4 (scalar append)
    (8, 8, 32, 1),       # block size 1
    (16, 2, 128, 16),    # head_dim 128 with group 8 -> generic kernel
], ids=["gate", "bs5", "g32", "hd256", "hd96", "hd5", "bs1", "g8"])
def test_generic_kernel(H, KV, hd, bs, split_keys):
    split_keys(64)
    lens = [0, 1, bs - 1, bs, 63, 64, 65, 200]
    lens = [max(0, x) for x in lens]
    run_case(H, KV, hd, bs, lens, [1, 2, 1, 5, 1, 1, 9, 1], seed=hd + bs)


@pytest.mark.gpu
def test_first_token_is_its_value_row():
    """total_k = 1: the only key gets weight 1, so out equals the new V row
    exactly (the single-key closed form)."""
    H, KV, hd = 32, 8, 128
    pool = GpuPool(4, 1, KV * hd, 16, max_seqs=2, max_blocks=2)
    try:
        s = pool.new_seq(16)
        Q = torch.randn(1, H * hd, device="cuda")
        K = torch.randn(1, KV * hd, device="cuda")
        V = torch.randn(1, KV * hd, device="cuda")
        pkv.check(pkv.pkv_ensure_append(s, 1))
        out = torch.empty(1, H * hd, device="cuda")
        pkv.check(pkv.pkv_attn_with_paged(Q, K, V, 1, H, KV, hd, s, 0, 1, 0.1, out))
        exp = V.view(KV, 1, hd).expand(KV, H // KV, hd).reshape(1, H * hd)
        assert bits_equal(out, exp)
    finally:
        pool.close()


@pytest.mark.gpu
def test_block_permutation_invariance(split_keys):
    """Paging is storage only: the same histories in a shuffled and in an
    ordered pool give the same bits."""
    split_keys(128)
    a = run_case(32, 8, 128, 16, [40, 300, 999], [1, 1, 4], seed=3, shuffle=True,
                 check_m1=False, check_contig=False)
    b = run_case(32, 8, 128, 16, [40, 300, 999], [1, 1, 4], seed=3, shuffle=False,
                 check_m1=False, check_contig=False)
    assert bits_equal(a, b)


@pytest.mark.gpu
def test_multilayer_pool_layer_offsets(split_keys):
    split_keys(64)
    run_case(32, 8, 128, 16, [100, 17], [1, 2], n_layers=3, layer=2, seed=5)
    run_case(4, 2, 8, 4, [9, 3], [1, 3], n_layers=2, layer=1, seed=6)


@pytest.mark.gpu
def test_host_buffer_entry_point_matches_device_path():
    H, KV, hd, bs = 32, 8, 128, 16
    pool = GpuPool(64, 1, KV * hd, bs, max_seqs=4, max_blocks=32)
    try:
        seqs = [pool.new_seq(400) for _ in range(3)]
        for s, p in zip(seqs, [10, 100, 300]):
            pool.grow(s, p)
            pool.write_history(s, 0, torch.randn(p, KV * hd), torch.randn(p, KV * hd))
        nq = [1, 1, 2]
        Q = torch.randn(4, H * hd).pin_memory()
        K = torch.randn(4, KV * hd).pin_memory()
        V = torch.randn(4, KV * hd).pin_memory()
        pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
        out_h = torch.empty(4, H * hd).pin_memory()
        pkv.check(pkv.pkv_attn_batch_host(seqs, nq, Q, K, V, H, KV, hd, 0, 1, 0.088, out_h))
        out_d = torch.empty(4, H * hd, device="cuda")
        pkv.check(pkv.pkv_attn_batch(seqs, nq, Q.cuda(), K.cuda(), V.cuda(), H, KV, hd, 0, 1, 0.088,
                                     out_d))
        assert bits_equal(out_h.cuda(), out_d)
    finally:
        pool.close()


@pytest.mark.gpu
@pytest.mark.parametrize("pinned,decode_only", [(True, False), (False, False), (True, True)],
                         ids=["pinned", "pageable", "pinned-decode"])
def test_host_buffers_match_device_path_large_batch(pinned, decode_only):
    """Host-buffer calls: a ~75 MB batch of chunked-prefill rows and a run of
    20 forks that share a 2048-token prefix (one shared-prefix pass), or the
    forks and the other sequences' decode rows alone.  Page-locked buffers
    let the kernels use Q and out in host memory for decode calls (out only
    with a shared-prefix run); pageable ones, and calls with prefill rows,
    copy through device staging.  Every row equals the device-path call, bit
    for bit."""
    H, KV, hd, bs = 32, 8, 128, 16
    q_dim, kv_dim = H * hd, KV * hd
    g = torch.Generator().manual_seed(21)
    pool = GpuPool(1024, 1, kv_dim, bs, max_seqs=32, max_blocks=160, shuffle_seed=5)
    try:
        a = pool.new_seq(1024 + 256)
        pool.grow(a, 256)
        pool.write_history(a, 0, torch.randn(256, kv_dim, generator=g), torch.randn(256, kv_dim, generator=g))
        root = pool.new_seq(2048 + 8)
        pool.grow(root, 2048)
        pool.write_history(root, 0, torch.randn(2048, kv_dim, generator=g), torch.randn(2048, kv_dim, generator=g))
        forks = [pkv.pkv_seq_fork(root) for _ in range(20)]
        assert all(forks)
        b = pool.new_seq(1024 + 512)
        pool.grow(b, 512)
        pool.write_history(b, 0, torch.randn(512, kv_dim, generator=g), torch.randn(512, kv_dim, generator=g))
        c = pool.new_seq(1024)
        seqs = [a] + forks + [b, c]
        nq = [1] * 23 if decode_only else [1024] + [1] * 20 + [1024, 1024]
        T = sum(nq)
        Q = torch.randn(T, q_dim, generator=g)
        K = torch.randn(T, kv_dim, generator=g)
        V = torch.randn(T, kv_dim, generator=g)
        out_h = torch.full((T, q_dim), float("nan"))
        if pinned:
            Q, K, V, out_h = Q.pin_memory(), K.pin_memory(), V.pin_memory(), out_h.pin_memory()
            args = (Q, K, V, out_h)
        else:
            args = tuple(np.ascontiguousarray(t.numpy()) for t in (Q, K, V, out_h))
        pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
        pkv.check(pkv.pkv_attn_batch_host(seqs, nq, args[0], args[1], args[2], H, KV, hd, 0, 1, 0.088,
                                          args[3]))
        got = torch.from_numpy(args[3]) if not pinned else out_h
        out_d = torch.empty(T, q_dim, device="cuda")
        pkv.check(pkv.pkv_attn_batch(seqs, nq, Q.cuda(), K.cuda(), V.cuda(), H, KV, hd, 0, 1, 0.088,
                                     out_d))
        assert pkv.pkv_pool_last_work(pool.p)["prefix_tiles"] > 0     # the forks ran as one run
        pool.check_no_device_error()
        assert bits_equal(got.cuda(), out_d)
    finally:
        pool.close()


@pytest.mark.gpu
def test_error_paths_change_nothing():
    H, KV, hd, bs = 32, 8, 128, 16
    pool = GpuPool(8, 1, KV * hd, bs, max_seqs=4, max_blocks=8)
    try:
        a = pool.new_seq(64)
        Q = torch.randn(2, H * hd, device="cuda")
        K = torch.randn(2, KV * hd, device="cuda")
        out = torch.empty(2, H * hd, device="cuda")
        # rows not ensured
        assert pkv.pkv_attn_with_paged(Q, K, K, 1, H, KV, hd, a, 0, 1, 1.0, out) == pkv.PKV_ERR_SEQ
        pkv.check(pkv.pkv_ensure_append(a, 1))
        assert pkv.pkv_attn_with_paged(Q, K, K, 0, H, KV, hd, a, 0, 1, 1.0, out) == pkv.PKV_ERR_BAD_DIM
        assert pkv.pkv_attn_with_paged(Q, K, K, 1, 30, KV, hd, a, 0, 1, 1.0, out) == pkv.PKV_ERR_BAD_GQA
        assert pkv.pkv_attn_with_paged(Q, K, K, 1, H, KV, hd, None, 0, 1, 1.0, out) == pkv.PKV_ERR_SEQ
        assert pkv.pkv_attn_with_paged(Q, K, K, 1, H, KV, 64, a, 0, 1, 1.0, out) == pkv.PKV_ERR_BAD_DIM
        assert pkv.pkv_attn_with_paged(Q, K, K, 1, H, KV, hd, a, 1, 1, 1.0, out) == pkv.PKV_ERR_ARG
        assert pkv.pkv_attn_batch([a, a], [1, 1], Q, K, K, H, KV, hd, 0, 1, 1.0, out) == pkv.PKV_ERR_ARG
        mis = torch.empty(H * hd + 1, device="cuda")[1:].view(1, H * hd)
        assert pkv.pkv_attn_with_paged(mis, K, K, 1, H, KV, hd, a, 0, 1, 1.0, out) == pkv.PKV_ERR_ARG
        # shared block not privatised -> refused, not written
        pkv.check(pkv.pkv_attn_with_paged(Q[:1], K[:1], K[:1], 1, H, KV, hd, a, 0, 1, 1.0, out))
        pkv.check(pkv.pkv_advance(a, 1))
        b = pkv.pkv_seq_fork(a)
        assert pkv.pkv_attn_with_paged(Q[:1], K[:1], K[:1], 1, H, KV, hd, b, 0, 1, 1.0, out) == pkv.PKV_ERR_SEQ
        pool.check_no_device_error()
    finally:
        pool.close()


@pytest.mark.gpu
def test_launch_accounting_and_profiling():
    H, KV, hd = 32, 8, 128
    pool = GpuPool(64, 1, KV * hd, 16, max_seqs=4, max_blocks=64)
    try:
        s = pool.new_seq(1024)
        pool.grow(s, 900)
        pool.write_history(s, 0, torch.randn(900, KV * hd), torch.randn(900, KV * hd))
        pkv.check(pkv.pkv_ensure_append(s, 1))
        Q = torch.randn(1, H * hd, device="cuda")
        K = torch.randn(1, KV * hd, device="cuda")
        out = torch.empty(1, H * hd, device="cuda")
        pkv.pkv_profile_reset()
        pkv.pkv_profile_enable(True)
        n0 = pkv.pkv_launch_count()
        pkv.check(pkv.pkv_attn_with_paged(Q, K, K, 1, H, KV, hd, s, 0, 1, 0.1, out))
        torch.cuda.synchronize()
        pkv.pkv_profile_enable(False)
        n = pkv.pkv_launch_count() - n0
        kinds = {k: pkv.pkv_profile_read(k) for k in range(pkv.PKV_KERNEL_KINDS)}
        assert sum(v[1] for v in kinds.values()) == n
        # one prep launch (page table + append + counters) and one decode launch;
        # decode splits are merged inside the decode kernel
        assert n == 2
        assert kinds[pkv.PKV_KERNEL_DECODE][1] == 1 and kinds[pkv.PKV_KERNEL_DECODE][0] > 0
        assert kinds[pkv.PKV_KERNEL_APPEND][1] == 1
        assert kinds[pkv.PKV_KERNEL_MERGE][1] == 0
    finally:
        pkv.pkv_profile_reset()
        pool.close()


@pytest.mark.gpu
@pytest.mark.parametrize("H,KV", [(32, 8), (16, 8), (8, 8), (64, 8)], ids=["g4", "g2", "g1", "g8"])
def test_prefill_tensor_core_rows(H, KV, split_keys):
    """Rows with n_q >= 32 take the tcgen05 kind::f16 kernel: tiles of 128/G
    tokens, ragged last tiles, an empty history, and rows long enough to be
    cut into several key splits (split size 16 x 32 = 512 keys) and merged."""
    split_keys(32)
    run_case(H, KV, 128, 16, [0, 5, 31, 600, 1100], [32, 33, 100, 64, 47], seed=H + 1)


@pytest.mark.gpu
def test_prefill_noncausal_and_odd_blocks(split_keys):
    split_keys(512)
    run_case(32, 8, 128, 5, [0, 77, 300], [40, 96, 33], causal=0, seed=21)
    run_case(32, 8, 128, 4, [13, 250], [64, 50], causal=1, seed=22)


@pytest.mark.gpu
def test_prefill_and_decode_rows_in_one_batch(split_keys):
    """A batch mixing decode rows, short chunks (decode kernel) and long
    chunks (tensor-core kernel); every row equals its M = 1 launch."""
    split_keys(128)
    run_case(32, 8, 128, 16, [3000, 10, 257, 0, 999, 64], [1, 31, 32, 200, 1, 130], seed=23)


@pytest.mark.gpu
def test_prefill_rescales_diverge_within_a_warp(split_keys):
    """Scores that jump up by ~9.5 (base 2) at position 400 for half of the
    query heads and down for the other half: the rising rows move their
    reference max and rescale the TMEM accumulator while their neighbours in
    the same warp do not."""
    split_keys(512)
    H, KV, hd = 32, 8, 128

    def shape(kind, a, start):
        a = a.copy()
        if kind == "K":
            pos = start + np.arange(a.shape[0])
            step = np.where(pos < 400, -0.3, 0.28).astype(np.float32)[:, None]
            return (0.1 * a + step).astype(np.float32)
        q = a.reshape(a.shape[0], H, hd)
        sign = np.where(np.arange(H) % 2 == 0, 1.0, -1.0).astype(np.float32)[None, :, None]
        return (0.1 * q + sign).reshape(a.shape).astype(np.float32)

    run_case(H, KV, hd, 16, [900, 300], [64, 40], seed=31, shape_data=shape)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float8_e4m3fn], ids=["bf16", "fp8"])
def test_host_buffers_narrow_pools(dtype):
    """Decode rows on bf16 / fp8 pools through page-locked host buffers (the
    narrow-pool kernel reads Q and writes out in host memory, and takes the
    fused append) equal the device-path call on an identical pool, bit for
    bit, pool bytes included."""
    H, KV, hd, bs = 32, 8, 128, 16
    q_dim, kv_dim = H * hd, KV * hd
    lens = [5, 700, 1500, 2100, 33]

    def run(host):
        g = torch.Generator().manual_seed(8)
        pool = GpuPool(512, 1, kv_dim, bs, max_seqs=8, max_blocks=160, shuffle_seed=4, dtype=dtype)
        try:
            seqs = []
            for L in lens:
                s = pool.new_seq(L + 4)
                pool.grow(s, L)
                pool.write_history(s, 0, torch.randn(L, kv_dim, generator=g), torch.randn(L, kv_dim, generator=g))
                seqs.append(s)
            nq = [1] * len(lens)
            T = len(lens)
            Q, K, V = (torch.randn(T, d, generator=g) for d in (q_dim, kv_dim, kv_dim))
            pkv.check(pkv.pkv_ensure_append_batch(seqs, nq))
            if host:
                out = torch.full((T, q_dim), float("nan")).pin_memory()
                pkv.check(pkv.pkv_attn_batch_host(seqs, nq, Q.pin_memory(), K.pin_memory(), V.pin_memory(),
                                                  H, KV, hd, 0, 1, hd ** -0.5, out))
                out = out.cuda()
            else:
                out = torch.empty(T, q_dim, device="cuda")
                pkv.check(pkv.pkv_attn_batch(seqs, nq, Q.cuda(), K.cuda(), V.cuda(), H, KV, hd, 0, 1,
                                             hd ** -0.5, out))
            pool.check_no_device_error()
            torch.cuda.synchronize()
            return out, pool.K.view(torch.uint8).clone(), pool.V.view(torch.uint8).clone()
        finally:
            pool.close()

    oh, kh, vh = run(True)
    od, kd, vd = run(False)
    assert bits_equal(oh, od)
    assert torch.equal(kh, kd) and torch.equal(vh, vd)
