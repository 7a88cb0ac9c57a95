"""The paged-KV gate on the GPU ("nx_paged_kv_gate.nx source").

EQUIV  three rounds (5-token prefill, 1-token decode, 3-token chunk) x 2 layers:
       the paged path equals the contiguous twin bit for bit, and the oracle
       within tolerance.
FORK   fork after the prefill; both forks diverge by 2 tokens; copy-on-append
       fires and both forks equal fresh contiguous replays of their histories.
REWIND truncate fork A back to the fork point and append B's rows: A's outputs
       equal B's bit for bit (the speculative-decode rewind contract).

Block size 4 is the gate's own setting for the pool; block size 8 puts the
5-token prompt in one partial block, where the gate's literal checks on
pt[0] (diverged, refcount 1 each) apply verbatim.  At block size 4 only the
written tail block is copied and the full prefix block stays shared.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from synth import gate_inputs
from gpu_helpers import GpuPool, assert_close, bits_equal, contiguous_attend

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
G = json.load(open(os.path.join(GOLDEN, "gate_constants.json")))
NL, H, KV, HD = G["n_layers"], G["n_heads"], G["n_kv_heads"], G["head_dim"]
QD, KVD = H * HD, KV * HD
SCALE = G["scale"]


def cuda(a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.float32).cuda()


class ContigGpu:
    """Contiguous per-layer history on the device, appended by torch copies."""

    def __init__(self):
        self.K = torch.zeros(NL, 64, KVD, device="cuda")
        self.V = torch.zeros(NL, 64, KVD, device="cuda")
        self.len = 0

    def attn(self, Q, K, V, n, layer):
        self.K[layer, self.len:self.len + n] = cuda(K)
        self.V[layer, self.len:self.len + n] = cuda(V)
        tk = self.len + n
        return contiguous_attend(cuda(Q), self.K[layer, :tk], self.V[layer, :tk], n, tk, H, KV, HD,
                                 1, SCALE)

    def advance(self, n):
        self.len += n


def paged_round(pool, seq, Q, K, V, n):
    """ensure once, append + attend per layer, advance once; outputs per layer."""
    assert pkv.pkv_ensure_append(seq, n) == 0, pkv.pkv_last_error()
    outs = []
    for layer in range(NL):
        out = torch.empty(n, QD, device="cuda")
        rc = pkv.pkv_attn_with_paged(cuda(Q), cuda(K), cuda(V), n, H, KV, HD, seq, layer, 1, SCALE,
                                     out)
        assert rc == 0, pkv.pkv_last_error()
        outs.append(out)
    assert pkv.pkv_advance(seq, n) == 0
    return torch.stack(outs)


def contig_round(cc, Q, K, V, n):
    outs = [cc.attn(Q, K, V, n, layer) for layer in range(NL)]
    cc.advance(n)
    return torch.stack(outs)


def oracle_round(oc, Q, K, V, n):
    outs = []
    for layer in range(NL):
        rc, o = oc.attn_with_cache(Q, K, V, n, H, KV, HD, layer, 1, SCALE)
        assert rc == 0
        outs.append(o)
    oc.advance(n)
    return np.stack(outs)


@pytest.mark.gpu
def test_gate_kat_on_device_pool():
    g = json.load(open(os.path.join(GOLDEN, "pool_kat.json")))
    pool = GpuPool(g["n_blocks"], NL, KVD, 4, max_seqs=4, max_blocks=16)
    try:
        assert [pkv.pkv_alloc_block(pool.p) for _ in g["allocs"]] == g["allocs"]
        assert pkv.pkv_unref_block(pool.p, g["release"]) == 0
        assert pkv.pkv_alloc_block(pool.p) == g["realloc"]
    finally:
        pool.close()


@pytest.mark.gpu
@pytest.mark.parametrize("bs", [4, 8])
def test_gate_equiv(bs):
    x = gate_inputs(G["seed"])
    pool = GpuPool(16, NL, KVD, bs, max_seqs=4, max_blocks=64 // bs)
    try:
        s = pool.new_seq(64)
        cc = ContigGpu()
        oc = oracle.ContiguousCache(NL, KV, 64, HD)
        vmax = 8.0
        for name, n in zip(("1", "2", "3"), G["rounds"]):
            Q, K, V = x["Q" + name], x["K" + name], x["V" + name]
            op = paged_round(pool, s, Q, K, V, n)
            ocg = contig_round(cc, Q, K, V, n)
            assert bits_equal(op, ocg), "paged != contiguous in round " + name
            assert_close(op.cpu().numpy(), oracle_round(oc, Q, K, V, n), vmax, "round " + name)
        pool.check_no_device_error()
    finally:
        pool.close()


@pytest.mark.gpu
@pytest.mark.parametrize("bs", [4, 8])
def test_gate_fork_cow_and_rewind(bs):
    x = gate_inputs(G["seed"])
    pool = GpuPool(16, NL, KVD, bs, max_seqs=4, max_blocks=64 // bs)
    try:
        fA = pool.new_seq(64)
        paged_round(pool, fA, x["Q1"], x["K1"], x["V1"], 5)
        fB = pkv.pkv_seq_fork(fA)
        assert fB
        pa = pkv.pkv_seq_page_table(fA)
        assert pkv.pkv_refcnt(pool.p, pa[0]) == 2       # shared prompt block

        opA = paged_round(pool, fA, x["QA"], x["KA"], x["VA"], 2)
        opB = paged_round(pool, fB, x["QB"], x["KB"], x["VB"], 2)
        pa, pb = pkv.pkv_seq_page_table(fA), pkv.pkv_seq_page_table(fB)
        tail = (G["fork_after"] - 1) // bs
        assert pa[tail] != pb[tail]
        assert pkv.pkv_refcnt(pool.p, pa[tail]) == 1 and pkv.pkv_refcnt(pool.p, pb[tail]) == 1
        if bs == 8:
            assert pa[0] != pb[0]
        else:
            assert pa[0] == pb[0] and pkv.pkv_refcnt(pool.p, pa[0]) == 2

        # ground truth: fresh contiguous replays of both histories
        for Qd, Kd, Vd, op in (("QA", "KA", "VA", opA), ("QB", "KB", "VB", opB)):
            cc = ContigGpu()
            contig_round(cc, x["Q1"], x["K1"], x["V1"], 5)
            ref = contig_round(cc, x[Qd], x[Kd], x[Vd], 2)
            assert bits_equal(op, ref)
            oc = oracle.ContiguousCache(NL, KV, 64, HD)
            oracle_round(oc, x["Q1"], x["K1"], x["V1"], 5)
            assert_close(op.cpu().numpy(), oracle_round(oc, x[Qd], x[Kd], x[Vd], 2), 8.0, Qd)

        # rewind A to the fork point, append B's rows: A now answers as B
        assert pkv.pkv_seq_truncate(fA, G["truncate_to"]) == 0
        opR = paged_round(pool, fA, x["QB"], x["KB"], x["VB"], 2)
        assert bits_equal(opR, opB)
        pool.check_no_device_error()
    finally:
        pool.close()


@pytest.mark.gpu
def test_gqa_selftest_on_gpu():
    """"nx_f32_gqa_attention.nx source", self-test: Q = 0 -> mean(V) = [4, 6] for
    both heads and both tokens; 3 query heads over 2 kv heads is rejected."""
    g = json.load(open(os.path.join(GOLDEN, "gqa_selftest.json")))
    n, hq, hk, hd = g["n_tokens"], g["n_q_heads"], g["n_kv_heads"], g["head_dim"]
    Q = cuda(np.array(g["Q"], np.float32).reshape(n, hq * hd))
    K = cuda(np.array(g["K"], np.float32).reshape(n, hk * hd))
    V = cuda(np.array(g["V"], np.float32).reshape(n, hk * hd))
    out = contiguous_attend(Q, K, V, n, n, hq, hk, hd, g["causal"], g["scale"])
    exp = np.broadcast_to(np.array(g["expected_per_head"], np.float32), (n, hq, hd))
    got = out.cpu().numpy().reshape(n, hq, hd)
    assert np.all(np.abs(got - exp) < g["tol"])
    bad = g["bad_grouping"]
    o2 = torch.empty(n, bad["n_q_heads"] * hd, device="cuda")
    rc = pkv.pkv_attn_contiguous(torch.zeros(n, bad["n_q_heads"] * hd, device="cuda"), K, V, n, n,
                                 bad["n_q_heads"], bad["n_kv_heads"], hd, 0, 1.0, o2, None)
    assert rc == pkv.PKV_ERR_BAD_GQA
