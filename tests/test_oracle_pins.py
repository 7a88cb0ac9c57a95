"""Pins for the attention oracle (CPU only).

Each check ties ``oracle.attend`` to something other than itself: the pages'
own worked example and rejection case ("nx_f32_gqa_attention.nx source",
self-test), closed forms (Q = 0 gives the mean of the visible value rows; a
single key returns its value row; two keys give a logistic weight), a library
routine (torch's scaled_dot_product_attention in float64 with the kv heads
expanded and an explicit offset-causal mask), and brute force at 40 digits on
tiny inputs.  ``test_mutations_are_caught`` recompiles the oracle with a
plausible mistake planted in each copy (wrong head map, off-by-one query
position, dropped scale or normaliser, flipped sign, misindexed operand) and
checks that the same battery rejects every one of them.
"""
import json
import math
import os
import shutil
import subprocess
import ctypes

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# the battery: every pin takes an ``attend`` callable with oracle.attend's API
# and raises AssertionError on failure


def pin_selftest(attend):
    g = _load_golden("gqa_selftest.json")
    rc, out = attend(g["Q"], g["K"], g["V"], g["n_tokens"], g["n_tokens"], g["n_q_heads"],
                     g["n_kv_heads"], g["head_dim"], g["causal"], g["scale"])
    assert rc == 0
    out = out.reshape(g["n_tokens"], g["n_q_heads"], g["head_dim"])
    exp = np.array(g["expected_per_head"], dtype=np.float64)
    assert np.all(np.abs(out - exp) < g["tol"])
    # mean of the integers 2,6 and 4,8 is exact in f32
    assert np.array_equal(out, np.broadcast_to(exp.astype(np.float32), out.shape))
    bad = g["bad_grouping"]
    rc, _ = attend(g["Q"], g["K"], g["V"], g["n_tokens"], g["n_tokens"], bad["n_q_heads"],
                   bad["n_kv_heads"], g["head_dim"], g["causal"], g["scale"])
    assert rc != 0


def pin_q_zero_mean(attend):
    """Q = 0: every score is 0, the softmax is uniform over the visible keys,
    and query i of a block of n_q sees keys 0..total_k-n_q+i (offset-causal).
    Each kv head carries different values, so a wrong head map shows."""
    rng = np.random.default_rng(1)
    for (n_q, past, H, KV, hd) in [(3, 4, 4, 2, 8), (1, 9, 6, 3, 4), (5, 0, 8, 2, 16)]:
        total_k = past + n_q
        V = rng.standard_normal((total_k, KV, hd)).astype(np.float32) + \
            np.arange(KV, dtype=np.float32)[None, :, None] * 10.0
        K = rng.standard_normal((total_k, KV * hd)).astype(np.float32)
        Q = np.zeros((n_q, H * hd), np.float32)
        rc, out = attend(Q, K, V.reshape(total_k, -1), n_q, total_k, H, KV, hd, 1, 0.3)
        assert rc == 0
        out = out.reshape(n_q, H, hd)
        g = H // KV
        for i in range(n_q):
            vis = total_k - n_q + i + 1
            for h in range(H):
                exp = V[:vis, h // g, :].astype(np.float64).mean(axis=0)
                np.testing.assert_allclose(out[i, h], exp, rtol=1e-6, atol=1e-6)


def pin_single_key(attend):
    """One key: the softmax weight is exactly 1 and out equals the value row."""
    rng = np.random.default_rng(2)
    H, KV, hd = 4, 2, 8
    Q = rng.standard_normal((1, H * hd)).astype(np.float32)
    K = rng.standard_normal((1, KV * hd)).astype(np.float32)
    V = rng.standard_normal((1, KV * hd)).astype(np.float32)
    rc, out = attend(Q, K, V, 1, 1, H, KV, hd, 1, 0.25)
    assert rc == 0
    out = out.reshape(H, hd)
    for h in range(H):
        assert np.array_equal(out[h], V.reshape(KV, hd)[h // 2])


def pin_two_keys(attend):
    """Two keys: out = (1-w) V0 + w V1 with w = 1 / (1 + exp(-scale (s1 - s0)))."""
    rng = np.random.default_rng(3)
    H, KV, hd, scale = 2, 1, 4, 0.37
    Q = rng.standard_normal((1, H * hd)).astype(np.float32)
    K = rng.standard_normal((2, KV * hd)).astype(np.float32)
    V = rng.standard_normal((2, KV * hd)).astype(np.float32)
    rc, out = attend(Q, K, V, 1, 2, H, KV, hd, 1, scale)
    assert rc == 0
    out = out.reshape(H, hd)
    for h in range(H):
        q = Q[0, h * hd:(h + 1) * hd].astype(np.float64)
        d = float(np.float32(scale)) * (q @ K[1].astype(np.float64) - q @ K[0].astype(np.float64))
        w = 1.0 / (1.0 + math.exp(-d))
        exp = (1 - w) * V[0].astype(np.float64) + w * V[1].astype(np.float64)
        np.testing.assert_allclose(out[h], exp, rtol=1e-6, atol=1e-7)


def _sdpa64(Q, K, V, n_q, total_k, H, KV, hd, causal, scale):
    torch = pytest.importorskip("torch")
    q = torch.tensor(Q, dtype=torch.float64).reshape(n_q, H, hd).transpose(0, 1)[None]
    k = torch.tensor(K, dtype=torch.float64).reshape(total_k, KV, hd).transpose(0, 1)
    v = torch.tensor(V, dtype=torch.float64).reshape(total_k, KV, hd).transpose(0, 1)
    k = k.repeat_interleave(H // KV, dim=0)[None]
    v = v.repeat_interleave(H // KV, dim=0)[None]
    i = torch.arange(n_q)[:, None]
    j = torch.arange(total_k)[None, :]
    mask = (j <= total_k - n_q + i) if causal else torch.ones(n_q, total_k, dtype=torch.bool)
    o = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=mask, scale=float(np.float32(scale)))
    return o[0].transpose(0, 1).reshape(n_q, H * hd).numpy()


def pin_sdpa_float64(attend):
    rng = np.random.default_rng(4)
    cases = [(1, 0, 4, 2, 8, 1), (3, 5, 4, 2, 8, 1), (7, 30, 8, 2, 16, 1), (4, 12, 6, 6, 4, 1),
             (5, 9, 8, 1, 32, 0), (2, 40, 32, 8, 128, 1), (9, 3, 4, 4, 8, 0), (6, 17, 12, 3, 64, 1)]
    for (n_q, past, H, KV, hd, causal) in cases:
        total_k = past + n_q
        scale = 1.0 / math.sqrt(hd)
        Q = rng.standard_normal((n_q, H * hd)).astype(np.float32)
        K = rng.standard_normal((total_k, KV * hd)).astype(np.float32)
        V = rng.standard_normal((total_k, KV * hd)).astype(np.float32)
        rc, out = attend(Q, K, V, n_q, total_k, H, KV, hd, causal, scale)
        assert rc == 0
        ref = _sdpa64(Q, K, V, n_q, total_k, H, KV, hd, causal, scale)
        np.testing.assert_allclose(out, ref, rtol=2e-7, atol=2e-7 * np.abs(V).max())


def pin_bruteforce_mp(attend):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    rng = np.random.default_rng(5)
    n_q, total_k, H, KV, hd, scale = 2, 4, 4, 2, 3, 0.7
    Q = rng.standard_normal((n_q, H * hd)).astype(np.float32)
    K = rng.standard_normal((total_k, KV * hd)).astype(np.float32)
    V = rng.standard_normal((total_k, KV * hd)).astype(np.float32)
    rc, out = attend(Q, K, V, n_q, total_k, H, KV, hd, 1, scale)
    assert rc == 0
    sc = mp.mpf(float(np.float32(scale)))
    for i in range(n_q):
        for h in range(H):
            kv = h // (H // KV)
            vis = total_k - n_q + i + 1
            s = [sc * mp.fsum(mp.mpf(float(Q[i, h * hd + d])) * mp.mpf(float(K[j, kv * hd + d]))
                              for d in range(hd)) for j in range(vis)]
            w = [mp.e ** x for x in s]
            den = mp.fsum(w)
            for d in range(hd):
                exact = mp.fsum(w[j] * mp.mpf(float(V[j, kv * hd + d])) for j in range(vis)) / den
                got = float(out[i, h * hd + d])
                # correctly rounded to f32 up to the double-precision stages
                assert abs(got - float(exact)) <= float(np.spacing(np.float32(abs(float(exact))))) + 1e-12


def pin_causal_flag(attend):
    """causal=0 sees every key; the last query of a block sees every key
    either way, the earlier ones differ."""
    rng = np.random.default_rng(6)
    n_q, total_k, H, KV, hd = 4, 10, 4, 2, 8
    Q = rng.standard_normal((n_q, H * hd)).astype(np.float32)
    K = rng.standard_normal((total_k, KV * hd)).astype(np.float32)
    V = rng.standard_normal((total_k, KV * hd)).astype(np.float32)
    _, oc = attend(Q, K, V, n_q, total_k, H, KV, hd, 1, 0.3)
    _, of = attend(Q, K, V, n_q, total_k, H, KV, hd, 0, 0.3)
    assert np.array_equal(oc[-1], of[-1])
    for i in range(n_q - 1):
        assert not np.allclose(oc[i], of[i])


BATTERY = [pin_selftest, pin_q_zero_mean, pin_single_key, pin_two_keys, pin_sdpa_float64,
           pin_bruteforce_mp, pin_causal_flag]


@pytest.mark.parametrize("pin", BATTERY, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.attend)


def test_bad_dims_and_grouping():
    z = np.zeros(64, np.float32)
    assert oracle.attend(z, z, z, 0, 1, 4, 2, 8, 1, 1.0)[0] == oracle.ERR_BAD_DIM
    assert oracle.attend(z, z, z, 1, 1, 0, 2, 8, 1, 1.0)[0] == oracle.ERR_BAD_DIM
    assert oracle.attend(z, z, z, 1, 1, 4, 0, 8, 1, 1.0)[0] == oracle.ERR_BAD_DIM
    assert oracle.attend(z, z, z, 1, 1, 4, 2, 0, 1, 1.0)[0] == oracle.ERR_BAD_DIM
    assert oracle.attend(z, z, z, 2, 1, 4, 2, 8, 1, 1.0)[0] == oracle.ERR_BAD_DIM
    assert oracle.attend(z, z, z, 1, 1, 3, 2, 4, 1, 1.0)[0] == oracle.ERR_BAD_GQA


# ---------------------------------------------------------------------------
# planted mistakes: each mutated copy of the oracle must fail the battery

MUTATIONS = {
    "head_map_modulo": ("const int kv_head = h / group;",
                        "const int kv_head = h % n_kv_heads;"),
    "q_pos_off_by_one": ("const int q_pos = total_k - n_q + i;",
                         "const int q_pos = total_k - n_q + i - 1 + (i == 0);"),
    "q_pos_not_offset": ("const int q_pos = total_k - n_q + i;", "const int q_pos = i;"),
    "scale_dropped": ("s[j] = (double)scale * dot;", "s[j] = dot;"),
    "scale_squared": ("s[j] = (double)scale * dot;", "s[j] = (double)scale * (double)scale * dot;"),
    "no_normaliser": ("o[d] = (float)(acc[d] / denom);", "o[d] = (float)(acc[d]);"),
    "sign_flipped": ("const double p = exp(s[j] - m);", "const double p = exp(m - s[j]);"),
    "diagonal_dropped": ("const int n_visible = causal ? q_pos + 1 : total_k;",
                         "const int n_visible = causal ? (q_pos > 0 ? q_pos : 1) : total_k;"),
    "v_rows_reversed": ("const float *v = V + (size_t)j * kv_dim",
                        "const float *v = V + (size_t)(n_visible - 1 - j) * kv_dim"),
    "k_head_wrong": ("const float *k = K + (size_t)j * kv_dim + (size_t)kv_head * head_dim;",
                     "const float *k = K + (size_t)j * kv_dim + (size_t)(n_kv_heads - 1 - kv_head) * head_dim;"),
    "k_dims_transposed": ("dot += (double)q[d] * (double)k[d];",
                          "dot += (double)q[d] * (double)k[head_dim - 1 - d];"),
}


def _mutant_attend(libpath):
    lib = ctypes.CDLL(libpath)
    fp = ctypes.POINTER(ctypes.c_float)
    lib.oracle_attend.argtypes = [fp, fp, fp] + [ctypes.c_int] * 6 + [ctypes.c_float, fp]
    lib.oracle_attend.restype = ctypes.c_int

    def attend(Q, K, V, n_q, total_k, n_heads, n_kv_heads, head_dim, causal, scale):
        Qa = np.ascontiguousarray(np.asarray(Q, np.float32).reshape(-1))
        Ka = np.ascontiguousarray(np.asarray(K, np.float32).reshape(-1))
        Va = np.ascontiguousarray(np.asarray(V, np.float32).reshape(-1))
        q_dim = n_heads * head_dim
        out = np.zeros(max(1, n_q * q_dim), np.float32)
        p = lambda a: a.ctypes.data_as(fp)  # noqa: E731
        rc = lib.oracle_attend(p(Qa), p(Ka), p(Va), n_q, total_k, n_heads, n_kv_heads,
                               head_dim, causal, float(np.float32(scale)), p(out))
        return rc, (out[:n_q * q_dim].reshape(n_q, q_dim) if rc == 0 else None)
    return attend


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutations_are_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attention.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, "mutation anchor not found: " + old
    mutated = tmp_path / "attention_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(lib),
                           str(mutated), "-lm"])
    attend = _mutant_attend(str(lib))
    failures = 0
    for pin in BATTERY:
        try:
            with np.errstate(all="ignore"):
                pin(attend)
        except (AssertionError, ValueError, TypeError, FloatingPointError):
            failures += 1
    assert failures > 0, "planted mistake %s passed every pin" % name


def test_thread_count_does_not_change_bits():
    """Each (query, head) pair is computed by one thread in a fixed order, so
    the oracle gives the same bits on one thread and on every core."""
    rng = np.random.default_rng(11)
    n_q, tk, H, KV, hd = 7, 300, 8, 2, 16
    Q = rng.standard_normal((n_q, H * hd)).astype(np.float32)
    K = rng.standard_normal((tk, KV * hd)).astype(np.float32)
    V = rng.standard_normal((tk, KV * hd)).astype(np.float32)
    try:
        oracle.set_threads(1)
        rc1, o1 = oracle.attend(Q, K, V, n_q, tk, H, KV, hd, 1, 0.25)
        n = oracle.set_threads(0)
        rcn, on = oracle.attend(Q, K, V, n_q, tk, H, KV, hd, 1, 0.25)
    finally:
        oracle.set_threads(0)
    assert rc1 == rcn == 0 and n >= 1
    assert np.array_equal(o1, on)
