"""Device failures reach the caller as status codes.

The kernels never stop on a bad page-table entry or an expired wait: they
skip the access, or give up the tile, and OR a bit into a device error word
(PKV_DEVERR_BOUNDS, PKV_DEVERR_TIMEOUT).  pkv_sync_error (pool calls) and
pkv_contiguous_sync_error (the contiguous entry points) wait for the work,
read and clear the word and map it to PKV_ERR_DEVICE_BOUNDS /
PKV_ERR_DEVICE_TIMEOUT -- the fail-fast return codes of "nx_f32_attn_paged.nx
source" (the NX_F32_AP_* checks at the top of nx_f32_attn_with_paged),
carried over to failures found after a call returned.

No kernel is made to fail: the bits are set from the host with
pkv_debug_or_error_bits, exactly where a kernel would set them, and the
tests check the mapping, that reading clears the word, that the words gather
bits across calls until read, and that clean work reports PKV_OK.
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import GpuPool


def _contig_call(fn, n_q=1, tk=300, H=4, KV=2, hd=64):
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    Q = torch.randn(n_q, H * hd, device="cuda", generator=g)
    K = torch.randn(tk, KV * hd, device="cuda", generator=g)
    V = torch.randn(tk, KV * hd, device="cuda", generator=g)
    out = torch.empty(n_q, H * hd, device="cuda")
    rc = fn(Q, K, V, n_q, tk, H, KV, hd, 1, 1.0 / math.sqrt(hd), out, torch.cuda.current_stream())
    assert rc == pkv.PKV_OK, pkv.pkv_last_error()
    return out


@pytest.mark.gpu
def test_pool_error_word_mapping():
    pool = GpuPool(8, 1, 16, 4, max_seqs=2, max_blocks=4)
    try:
        assert pkv.pkv_sync_error(pool.p) == pkv.PKV_OK
        for bits, rc in ((pkv.PKV_DEVERR_BOUNDS, pkv.PKV_ERR_DEVICE_BOUNDS),
                         (pkv.PKV_DEVERR_TIMEOUT, pkv.PKV_ERR_DEVICE_TIMEOUT),
                         (pkv.PKV_DEVERR_BOUNDS | pkv.PKV_DEVERR_TIMEOUT, pkv.PKV_ERR_DEVICE_TIMEOUT)):
            assert pkv.pkv_debug_or_error_bits(pool.p, pkv.PKV_ERRWORD_POOL, bits) == pkv.PKV_OK
            assert pkv.pkv_sync_error(pool.p) == rc
            msg = pkv.pkv_last_error()
            if bits & pkv.PKV_DEVERR_TIMEOUT:
                assert "bounded wait" in msg
            if bits & pkv.PKV_DEVERR_BOUNDS:
                assert "out of range" in msg
            assert pkv.pkv_sync_error(pool.p) == pkv.PKV_OK     # reading cleared it
    finally:
        pool.close()


@pytest.mark.gpu
def test_contiguous_error_words_gather_until_read():
    s = torch.cuda.current_stream()
    _contig_call(pkv.pkv_attn_contiguous)
    _contig_call(pkv.pkv_attn_contiguous_noalloc)
    assert pkv.pkv_contiguous_sync_error(s) == pkv.PKV_OK
    # each word, each bit
    for which in (pkv.PKV_ERRWORD_CONTIGUOUS, pkv.PKV_ERRWORD_NOALLOC):
        for bits, rc in ((pkv.PKV_DEVERR_BOUNDS, pkv.PKV_ERR_DEVICE_BOUNDS),
                         (pkv.PKV_DEVERR_TIMEOUT, pkv.PKV_ERR_DEVICE_TIMEOUT)):
            assert pkv.pkv_debug_or_error_bits(None, which, bits) == pkv.PKV_OK
            assert pkv.pkv_contiguous_sync_error(s) == rc
            assert pkv.pkv_contiguous_sync_error(s) == pkv.PKV_OK
    # a bit set before clean calls is still there after them (no call clears it)
    assert pkv.pkv_debug_or_error_bits(None, pkv.PKV_ERRWORD_NOALLOC, pkv.PKV_DEVERR_BOUNDS) == 0
    assert pkv.pkv_debug_or_error_bits(None, pkv.PKV_ERRWORD_CONTIGUOUS, pkv.PKV_DEVERR_TIMEOUT) == 0
    _contig_call(pkv.pkv_attn_contiguous_noalloc)
    _contig_call(pkv.pkv_attn_contiguous)
    assert pkv.pkv_contiguous_sync_error(s) == pkv.PKV_ERR_DEVICE_TIMEOUT
    assert "out of range" in pkv.pkv_last_error()          # both words were read
    assert pkv.pkv_contiguous_sync_error(s) == pkv.PKV_OK


@pytest.mark.gpu
def test_error_bits_arguments_are_checked():
    assert pkv.pkv_debug_or_error_bits(None, pkv.PKV_ERRWORD_POOL, 1) == pkv.PKV_ERR_ARG
    assert pkv.pkv_debug_or_error_bits(None, 7, 1) == pkv.PKV_ERR_ARG
    assert pkv.pkv_debug_or_error_bits(None, pkv.PKV_ERRWORD_CONTIGUOUS, 4) == pkv.PKV_ERR_ARG
    host = pkv.pkv_pool_new(8, 1, 16, 4, None, None, 2, 4, None, pkv.PKV_POOL_HOST_ONLY)
    try:
        assert pkv.pkv_debug_or_error_bits(host, pkv.PKV_ERRWORD_POOL, 1) == pkv.PKV_ERR_ARG
    finally:
        pkv.pkv_pool_free(host)


@pytest.mark.gpu
def test_tf32_probe_reports_rates_and_checks_arguments():
    """The tcgen05 TF32 issue-rate probe: positive clocks per MMA and rate for
    both operand sources, wider MMAs no cheaper per flop than N = 64 pays in
    clocks, and bad arguments rejected before any launch."""
    for n, ts in ((64, True), (128, True), (64, False)):
        clk, tf = pkv.pkv_probe_tf32_mma(n, ts, 256)
        assert clk > 0 and tf > 0, (n, ts, clk, tf)
    c64, _ = pkv.pkv_probe_tf32_mma(64, True, 1024)
    c128, _ = pkv.pkv_probe_tf32_mma(128, True, 1024)
    assert c128 >= c64 * 0.9          # twice the work per MMA never costs less time
    for args in ((96, 1, 256), (64, 1, 100), (64, 1, 0)):
        with pytest.raises(pkv.PkvError):
            pkv.pkv_probe_tf32_mma(*args)


@pytest.mark.gpu
def test_f16_probe_reports_rates_and_checks_arguments():
    """The same for the kind::f16 probe (the prefill kernel's instruction):
    positive clocks and rates, and bad arguments rejected."""
    for n, ts in ((64, True), (128, True), (64, False)):
        clk, tf = pkv.pkv_probe_f16_mma(n, ts, 256)
        assert clk > 0 and tf > 0, (n, ts, clk, tf)
    c64, _ = pkv.pkv_probe_f16_mma(64, True, 1024)
    c128, _ = pkv.pkv_probe_f16_mma(128, True, 1024)
    assert c128 >= c64 * 0.9
    for args in ((96, 1, 256), (64, 1, 100), (64, 1, 0)):
        with pytest.raises(pkv.PkvError):
            pkv.pkv_probe_f16_mma(*args)
