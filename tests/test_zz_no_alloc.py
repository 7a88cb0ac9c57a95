"""pkv_attn_contiguous_noalloc: contiguous attention for callers that cannot
let a library allocate device memory (an engine that has reserved its whole
device-memory budget, code inside an allocator callback, loops where
cudaMalloc/cudaFree could synchronise the device).  Its scratch is one static
device array, so its output must match pkv_attn_contiguous -- the entry point
that allocates its scratch per call -- within the tests' tolerance, on calls
in a row (each finds the previous call's contents in the array), and the
oracle within the same tolerance.  The calls cover both kernels the entry
point dispatches: split-K decode (with split partials and their merge in the
array) and the tensor-core kernel for rows of 32 or more queries (its tiles'
descriptors, the split pass's operand images and the kernel's reads of them
in the array), the latter both before and after a call that left other
partials behind; and a 32-query row whose images would not fit in the array,
which goes to split-K decode instead.

This file is collected last so that a run stopping at the first failure has
run every other test before it; it also passes alone in a fresh process.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_nx_gb300 as pkv
from gpu_helpers import assert_close


def _case(n_q, past, H, KV, hd, causal, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    tk = past + n_q
    Q = torch.randn(n_q, H * hd, device="cuda", generator=g)
    Kc = torch.randn(tk, KV * hd, device="cuda", generator=g)
    Vc = torch.randn(tk, KV * hd, device="cuda", generator=g)
    scale = float(np.float32(1.0 / math.sqrt(hd)))
    return Q, Kc, Vc, n_q, tk, H, KV, hd, causal, scale


@pytest.mark.gpu
def test_no_alloc_matches_allocating_entry_point_on_two_calls():
    stream = torch.cuda.current_stream()
    cases = [
        _case(32, 16500, 32, 8, 128, 1, 4),  # images would not fit: split-K decode, splits + merge
        _case(1, 3000, 32, 8, 128, 1, 1),    # several splits + merge on the head_dim-128 kernel
        _case(64, 1024, 32, 8, 128, 1, 5),   # tensor-core kernel after stale decode partials
        _case(3, 40, 4, 2, 8, 1, 2),         # one split, generic kernel, stale scratch from call 1
        _case(40, 1500, 32, 8, 128, 0, 6),   # tensor-core kernel, non-causal, ragged tail, 12.6 MB of images
    ]
    for i, (Q, Kc, Vc, n_q, tk, H, KV, hd, causal, scale) in enumerate(cases):
        ref = torch.empty(n_q, H * hd, device="cuda")
        got = torch.full((n_q, H * hd), float("nan"), device="cuda")
        assert pkv.pkv_attn_contiguous(Q, Kc, Vc, n_q, tk, H, KV, hd, causal, scale, ref,
                                       stream) == pkv.PKV_OK, pkv.pkv_last_error()
        assert pkv.pkv_attn_contiguous_noalloc(Q, Kc, Vc, n_q, tk, H, KV, hd, causal, scale, got,
                                               stream) == pkv.PKV_OK, pkv.pkv_last_error()
        torch.cuda.synchronize()
        vmax = Vc.abs().max().item()
        assert_close(got.cpu().numpy(), ref.cpu().numpy(), vmax, "call %d" % i)
        rc, exp = oracle.attend(Q.cpu().numpy(), Kc.cpu().numpy(), Vc.cpu().numpy(), n_q, tk, H,
                                KV, hd, causal, scale)
        assert rc == 0
        assert_close(got.cpu().numpy(), exp, vmax, "call %d vs the oracle" % i)
    assert pkv.pkv_contiguous_sync_error(stream) == pkv.PKV_OK, pkv.pkv_last_error()


@pytest.mark.gpu
def test_no_alloc_rejects_requests_beyond_its_scratch():
    # 31 queries (the split-K decode path) over a 70 000-key history need about
    # 70 MB of split partials, far beyond the static array; the buffers are
    # full size so that nothing could be read out of bounds in any case
    Q, Kc, Vc, n_q, tk, H, KV, hd, causal, scale = _case(31, 70000, 32, 8, 128, 1, 3)
    out = torch.empty(n_q, H * hd, device="cuda")
    rc = pkv.pkv_attn_contiguous_noalloc(Q, Kc, Vc, n_q, tk, H, KV, hd, causal, scale, out,
                                         torch.cuda.current_stream())
    assert rc == pkv.PKV_ERR_CAPACITY
    assert "static array" in pkv.pkv_last_error()
