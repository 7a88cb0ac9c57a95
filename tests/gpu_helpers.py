"""Helpers for the GPU parity tests: device pools backed by torch tensors,
history writes that bypass the library's kernels, and the tolerance.

Histories are written into the pool with torch indexing (not through the
library), so the oracle receives the generator's values and never anything
the CUDA path produced; the rows a call appends go through the library.
"""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_gqa_nx_gb300 as pkv
from synth.workloads import release_order


def tolerance(vmax: float) -> float:
    """max |err| <= 1e-5 * max|V| + 1e-6 (f32 attention output)."""
    return 1e-5 * float(vmax) + 1e-6


def assert_close(got, exp, vmax, what=""):
    got = np.asarray(got, dtype=np.float64)
    exp = np.asarray(exp, dtype=np.float64)
    assert got.shape == exp.shape, (got.shape, exp.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    err = float(np.max(np.abs(got - exp))) if got.size else 0.0
    tol = tolerance(vmax)
    assert err <= tol, "%s: max |err| %.3e > tol %.3e" % (what, err, tol)
    return err


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32))


class GpuPool:
    """A library pool whose K/V storage is a pair of caller-owned torch tensors
    [n_blocks, n_layers, block_size, kv_dim], pre-filled with NaN so that a read
    of a row nobody wrote poisons the output."""

    def __init__(self, n_blocks, n_layers, kv_dim, bs, max_seqs=64, max_blocks=4096,
                 shuffle_seed=None, fill=float("nan"), dtype=torch.float32, kv_scale=1.0):
        self.n_blocks, self.n_layers, self.kv_dim, self.bs = n_blocks, n_layers, kv_dim, bs
        self.K = torch.full((n_blocks, n_layers, bs, kv_dim), fill, device="cuda",
                            dtype=torch.float32).to(dtype)
        self.V = torch.full_like(self.K, fill)
        self.stream = torch.cuda.current_stream()
        self.kv_scale = float(kv_scale)
        flags = (pkv.PKV_POOL_BF16 if dtype == torch.bfloat16 else
                 pkv.PKV_POOL_FP8 if dtype == torch.float8_e4m3fn else 0)
        self.p = pkv.pkv_pool_new(n_blocks, n_layers, kv_dim, bs, self.K, self.V, max_seqs,
                                  max_blocks, self.stream, flags)
        assert self.p, pkv.pkv_last_error()
        if self.kv_scale != 1.0:
            pkv.check(pkv.pkv_pool_set_kv_scale(self.p, self.kv_scale))
        if shuffle_seed is not None:
            ids = [pkv.pkv_alloc_block(self.p) for _ in range(n_blocks)]
            assert ids == list(range(n_blocks))
            for b in release_order(n_blocks, shuffle_seed):
                assert pkv.pkv_unref_block(self.p, int(b)) == 0

    def new_seq(self, max_tokens):
        s = pkv.pkv_seq_new(self.p, max_tokens)
        assert s, pkv.pkv_last_error()
        return s

    def grow(self, seq, n):
        """Commit n tokens of history (metadata only; data via write_history)."""
        pkv.check(pkv.pkv_ensure_append(seq, n))
        pkv.check(pkv.pkv_advance(seq, n))

    def write_history(self, seq, layer, K_hist: torch.Tensor, V_hist: torch.Tensor, start=0):
        """Write rows [start, start+L) of layer `layer` directly (torch indexing)."""
        L = K_hist.shape[0]
        pt = torch.tensor(pkv.pkv_seq_page_table(seq), device="cuda", dtype=torch.long)
        pos = torch.arange(start, start + L, device="cuda")
        blk = pt[pos // self.bs]
        off = pos % self.bs
        # a bf16 / fp8 pool stores torch's float32 -> bfloat16 / float8_e4m3fn cast
        # (nearest, ties to even) of x / scale
        s = self.kv_scale
        self.K[blk, layer, off] = (K_hist.to(device="cuda", dtype=torch.float32) / s).to(self.K.dtype)
        self.V[blk, layer, off] = (V_hist.to(device="cuda", dtype=torch.float32) / s).to(self.V.dtype)

    def read_history(self, seq, layer, L):
        """Rows [0, L) as stored (the pool's element type; times kv_scale to read)."""
        pt = torch.tensor(pkv.pkv_seq_page_table(seq), device="cuda", dtype=torch.long)
        pos = torch.arange(L, device="cuda")
        return self.K[pt[pos // self.bs], layer, pos % self.bs], self.V[pt[pos // self.bs], layer, pos % self.bs]

    def read_values(self, seq, layer, L):
        """Rows [0, L) as the kernels read them: float32, element * kv_scale."""
        K, V = self.read_history(seq, layer, L)
        return K.float() * self.kv_scale, V.float() * self.kv_scale

    def check_no_device_error(self):
        assert pkv.pkv_sync_error(self.p) == pkv.PKV_OK, pkv.pkv_last_error()

    def close(self):
        torch.cuda.synchronize()
        pkv.pkv_pool_free(self.p)
        self.p = None


def contiguous_attend(Q, Kc, Vc, n_q, total_k, H, KV, hd, causal, scale):
    """The library's contiguous twin on device tensors; returns out."""
    out = torch.empty(n_q, H * hd, device="cuda", dtype=torch.float32)
    rc = pkv.pkv_attn_contiguous(Q.contiguous(), Kc.contiguous(), Vc.contiguous(), n_q, total_k, H,
                                 KV, hd, causal, scale, out, torch.cuda.current_stream())
    assert rc == 0, pkv.pkv_last_error()
    return out
