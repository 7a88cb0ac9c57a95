"""Pins of the oracle's rotary position embedding (NeoX pairing), each tied to
something other than the oracle itself: worked values computed by hand from
the definition in "nx_f32_llama_v4b.nx source", Block section (RoPE step:
position = sequence length, build the cos/sin table, apply in NeoX form),
closed forms, and the group properties a rotation must have.  A swapped
pairing (adjacent instead of half-split), a wrong frequency exponent, a sign
error or Q and K rotated differently each fail one of them."""
import math

import numpy as np
import pytest

import oracle


def test_position_zero_is_the_identity():
    x = np.random.default_rng(0).standard_normal((3, 2 * 8))
    assert np.array_equal(oracle.rope_neox(x, [0, 0, 0], 8, 10000.0), x)


def test_worked_values_head_dim_4():
    # hd = 4: pairs (0, 2) turn by pos * 1 and (1, 3) by pos * base^(-1/2).
    # e0 at position 1 -> (cos 1, 0, sin 1, 0); e1 -> (0, cos .01, 0, sin .01)
    # for base 10000 (10000^(-1/2) = 0.01); e2 -> (-sin 1, 0, cos 1, 0).
    e = np.eye(4)
    y = oracle.rope_neox(e, [1, 1, 1, 1], 4, 10000.0)
    c1, s1 = math.cos(1.0), math.sin(1.0)
    c2, s2 = math.cos(0.01), math.sin(0.01)
    np.testing.assert_allclose(y[0], [c1, 0, s1, 0], atol=1e-15)
    np.testing.assert_allclose(y[1], [0, c2, 0, s2], atol=1e-15)
    np.testing.assert_allclose(y[2], [-s1, 0, c1, 0], atol=1e-15)
    np.testing.assert_allclose(y[3], [0, -s2, 0, c2], atol=1e-15)


def test_head_dim_2_is_a_plane_rotation_by_pos():
    # one pair, theta_0 = 1: the angle is the position itself
    for pos in (1, 5, 1000, 32767):
        y = oracle.rope_neox(np.array([[0.6, -0.8]]), [pos], 2, 500000.0)
        c, s = math.cos(pos), math.sin(pos)
        np.testing.assert_allclose(y[0], [0.6 * c + 0.8 * s, 0.6 * s - 0.8 * c], atol=1e-12)


def test_every_head_gets_the_same_rotation():
    rng = np.random.default_rng(1)
    h = rng.standard_normal((1, 16))
    y = oracle.rope_neox(np.tile(h, (1, 4)), [123], 16, 10000.0)
    for k in range(4):
        np.testing.assert_array_equal(y[0, 16 * k:16 * (k + 1)], y[0, :16])


def test_rotation_preserves_pair_norms_and_composes():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 64))
    pos = np.array([0, 3, 77, 1024, 30000])
    y = oracle.rope_neox(x, pos, 32, 10000.0)
    for h in range(2):
        a, b = x[:, 32 * h:32 * h + 16], x[:, 32 * h + 16:32 * h + 32]
        ya, yb = y[:, 32 * h:32 * h + 16], y[:, 32 * h + 16:32 * h + 32]
        np.testing.assert_allclose(ya ** 2 + yb ** 2, a ** 2 + b ** 2, rtol=1e-12)
    # turning by p then by q is turning by p + q; by -p undoes p
    z = oracle.rope_neox(oracle.rope_neox(x, pos, 32, 10000.0), 2 * pos, 32, 10000.0)
    np.testing.assert_allclose(z, oracle.rope_neox(x, 3 * pos, 32, 10000.0), atol=1e-10)
    np.testing.assert_allclose(oracle.rope_neox(y, -pos, 32, 10000.0), x, atol=1e-10)


def test_scores_depend_on_the_offset_only():
    # <R(m) q, R(n) k> = <R(m + c) q, R(n + c) k> for every shift c
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((1, 64)), rng.standard_normal((1, 64))
    ref = (oracle.rope_neox(q, [40], 64, 10000.0) @ oracle.rope_neox(k, [7], 64, 10000.0).T).item()
    for c in (1, 100, 5000):
        got = (oracle.rope_neox(q, [40 + c], 64, 10000.0) @ oracle.rope_neox(k, [7 + c], 64, 10000.0).T).item()
        assert got == pytest.approx(ref, abs=1e-10)


def test_attention_over_rotated_rows_is_shift_invariant():
    # the attention output over rotated queries and keys only sees relative
    # positions: shifting every position by c leaves it unchanged
    rng = np.random.default_rng(4)
    H, KV, hd, n = 4, 2, 16, 12
    Q = rng.standard_normal((1, H * hd)).astype(np.float32)
    K = rng.standard_normal((n, KV * hd)).astype(np.float32)
    V = rng.standard_normal((n, KV * hd)).astype(np.float32)
    outs = []
    for c in (0, 333):
        pos = np.arange(n) + c
        Qr = oracle.rope_neox(Q, [n - 1 + c], hd, 10000.0)
        Kr = oracle.rope_neox(K, pos, hd, 10000.0)
        rc, o = oracle.attend(Qr, Kr, V, 1, n, H, KV, hd, 1, 0.25)
        assert rc == 0
        outs.append(o)
    np.testing.assert_allclose(outs[0], outs[1], atol=2e-6)


def test_float32_form_agrees_with_the_definition():
    # the float32 carrying-out differs from the float64 definition only by
    # float32 rounding (a few ulps of the pair's magnitude), and is exact at
    # position 0
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 128)).astype(np.float32)
    pos = np.array([0, 1, 17, 999, 12345, 30000])
    y64 = oracle.rope_neox(x, pos, 64, 10000.0)
    y32 = oracle.rope_neox_f32(x, pos, 64, 10000.0)
    assert y32.dtype == np.float32
    mag = np.abs(x).max()
    assert np.max(np.abs(y32 - y64)) <= 4 * 2.0 ** -24 * 2 * mag
    np.testing.assert_array_equal(y32[0], x[0])
    # and a wrong pairing in the float32 form would not pass the worked values
    e = np.eye(4, dtype=np.float32)
    y = oracle.rope_neox_f32(e, [1] * 4, 4, 10000.0)
    np.testing.assert_allclose(y[0], [np.cos(1.0), 0, np.sin(1.0), 0], atol=1e-7)
