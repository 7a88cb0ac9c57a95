"""Pins of the oracle's bf16 rounding (the bf16 pool stores every K/V row
rounded once to the nearest bfloat16, ties to even; not on the pages): values
worked by hand from the binary32 layout, torch's own float32 -> bfloat16 cast
on the CPU (a library routine), and the invariants of a rounding."""
import numpy as np
import torch

import oracle


def test_worked_values():
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    cases = {
        1.0: 1.0,                                   # exact
        1.0 + ulp: 1.0 + ulp,                       # exact
        1.0 + ulp / 2: 1.0,                         # tie, kept part even -> down
        1.0 + 3 * ulp / 2: 1.0 + 2 * ulp,           # tie, kept part odd -> up
        1.0 + ulp / 2 + 2.0 ** -20: 1.0 + ulp,      # just above the tie -> up
        1.0 + ulp / 2 - 2.0 ** -20: 1.0,            # just below the tie -> down
        -(1.0 + 3 * ulp / 2): -(1.0 + 2 * ulp),     # sign is kept, magnitude rounds
        # 3e38 = 1.7632.. * 2^127; 1.7632.. * 128 = 225.69 -> 226
        3.0e38: 226.0 / 128.0 * 2.0 ** 127,
        0.0: 0.0,
    }
    x = np.array(list(cases), dtype=np.float32)
    got = oracle.round_bf16(x)
    exp = np.array(list(cases.values()), dtype=np.float32)
    np.testing.assert_array_equal(got, exp)


def test_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000), rng.standard_normal(1000) * 1e30,
                        rng.standard_normal(1000) * 1e-30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), ref)


def test_rounding_invariants():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(10000).astype(np.float32)
    r = oracle.round_bf16(x)
    # idempotent, low 16 bits clear, within half a bf16 ulp, monotone
    np.testing.assert_array_equal(oracle.round_bf16(r), r)
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)
    ulp = np.spacing(np.abs(x)) * 2.0 ** 16
    assert np.all(np.abs(r.astype(np.float64) - x) <= ulp / 2)
    s = np.sort(x)
    assert np.all(np.diff(oracle.round_bf16(s)) >= 0)


# ---------------------------------------------------------------- fp8 e4m3 --

def test_e4m3_worked_values():
    # spacing 2^-3 in [1, 2), 2^5 in [256, 448]; subnormals m * 2^-9
    cases = {
        1.0: 1.0, 1.125: 1.125,
        1.0625: 1.0,                  # tie, kept mantissa 000 even -> down
        1.1875: 1.25,                 # tie, kept mantissa 001 odd -> up
        1.0625 + 2.0 ** -12: 1.125,   # just above the tie
        -1.1875: -1.25,
        448.0: 448.0,
        464.0: 448.0,                 # tie between 448 (even) and 480 (beyond range)
        500.0: 448.0, -1e6: -448.0,   # saturation
        2.0 ** -9: 2.0 ** -9,         # smallest subnormal
        2.0 ** -10: 0.0,              # tie between 0 (even) and 2^-9
        3 * 2.0 ** -10: 2.0 ** -8,    # tie between 2^-9 (odd) and 2 * 2^-9
        2.0 ** -6: 2.0 ** -6,         # smallest normal
        0.0: 0.0,
    }
    x = np.array(list(cases), dtype=np.float32)
    np.testing.assert_array_equal(oracle.round_e4m3(x), np.array(list(cases.values()), dtype=np.float32))


def test_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(100000) * 4, rng.uniform(-460, 460, 10000),
                        rng.standard_normal(1000) * 2e-3]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    np.testing.assert_array_equal(oracle.round_e4m3(x), ref)


def test_e4m3_scale_and_invariants():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(20000).astype(np.float32) * 20
    # a power-of-two scale is exact: e4m3(x / s) * s == round(x / s) * s
    for s in (0.25, 1.0, 8.0):
        np.testing.assert_array_equal(oracle.round_e4m3(x, s), oracle.round_e4m3(x / s) * s)
    r = oracle.round_e4m3(x)
    np.testing.assert_array_equal(oracle.round_e4m3(r), r)          # idempotent
    assert np.all(np.abs(r) <= 448)
    s = np.sort(x)
    assert np.all(np.diff(oracle.round_e4m3(s)) >= 0)               # monotone
    ok = np.abs(x) < 448
    rel = np.abs(r[ok].astype(np.float64) - x[ok]) / np.maximum(np.abs(x[ok]), 2.0 ** -6)
    assert rel.max() <= 2.0 ** -4 + 1e-12                           # half a step of 3 mantissa bits
    try:
        oracle.round_e4m3(x, 3.0)
        raise AssertionError("non-power-of-two scale accepted")
    except ValueError:
        pass
