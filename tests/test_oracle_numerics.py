"""Pins for the oracle's bfloat16 rounding against torch's float32 -> bfloat16 conversion
(an independent implementation of the same IEEE-style rounding) and hand-worked ties."""
import numpy as np
import torch

from oracle.numerics import to_bf16


def _torch_bf16(x32):
    return torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()


def test_matches_torch_on_float32_values_across_the_exponent_range():
    rng = np.random.default_rng(0)
    # random bit patterns: every exponent, subnormals, both signs (NaN/inf dropped)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    x32 = bits.view(np.float32)
    x32 = x32[np.isfinite(x32)]
    got = to_bf16(x32.astype(np.float64))
    want = _torch_bf16(x32)
    assert np.array_equal(got, want)
    # values near ties: the low 16 bits close to 0x8000
    hi = rng.integers(0, 2 ** 16, 20000, dtype=np.uint64).astype(np.uint32) << np.uint32(16)
    lo = (np.uint32(0x8000) + rng.integers(-2, 3, 20000).astype(np.int64)).astype(np.uint32)
    y32 = (hi | lo).view(np.float32)
    y32 = y32[np.isfinite(y32)]
    assert np.array_equal(to_bf16(y32.astype(np.float64)), _torch_bf16(y32))


def test_hand_worked_ties_and_edges():
    cases = {
        1.0 + 2.0 ** -8: 1.0,                         # tie, even neighbour is 1.0
        1.0 + 3 * 2.0 ** -8: 1.0 + 2.0 ** -6,         # tie, even neighbour is the upper one
        1.0 + 2.0 ** -8 + 2.0 ** -30: 1.0 + 2.0 ** -7,  # just above the tie
        -(1.0 + 2.0 ** -8): -1.0,
        2.0 ** -133: 2.0 ** -133,                     # smallest subnormal
        2.0 ** -134: 0.0,                             # tie with 0: even is 0
        3 * 2.0 ** -134: 2.0 ** -132,                 # tie between 1 and 2 units: even is 2
        255.5 * 2.0 ** -8: 1.0,                       # carries into the next exponent
        2.0 ** 128 - 2.0 ** 120: 2.0 ** 128 - 2.0 ** 120,   # largest finite
        2.0 ** 128 - 2.0 ** 119: np.inf,              # the overflow midpoint
        0.0: 0.0,
    }
    x = np.array(list(cases.keys()))
    np.testing.assert_array_equal(to_bf16(x), np.array(list(cases.values())))
