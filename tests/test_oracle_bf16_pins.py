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
