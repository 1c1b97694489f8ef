"""Pins for the oracle's round-to-nearest-even conversions.

The bfloat16 rounding is checked against PyTorch's CPU float32->bfloat16
conversion (a library routine) and, for doubles that float32 cannot hold,
against brute force in exact rational arithmetic.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import numeric


def _torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(x32.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # f32 subnormals
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 3.3895314e38,
                  np.inf, -np.inf, 1.17549435e-38, 1e-45], dtype=np.float32),
        # exact ties: 1 + 2^-8 (to even: 1), 1 + 3*2^-8 (to even: up)
        np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8)], dtype=np.float32),
    ])
    ours = numeric.f64_to_bf16_bits(x.astype(np.float64))
    ref = _torch_bf16_bits(x)
    np.testing.assert_array_equal(ours, ref)


def test_bf16_nan_stays_nan():
    bits = numeric.f64_to_bf16_bits(np.array([np.nan, -np.nan]))
    assert np.isnan(numeric.bf16_bits_to_f64(bits)).all()


def _bf16_values_exact():
    """Every finite positive bfloat16 value as an exact Fraction, sorted."""
    vals = []
    for b in range(0x0000, 0x7F80):
        f = np.array([b << 16], dtype=np.uint32).view(np.float32)[0]
        vals.append(Fraction(float(f)))
    return vals


def test_bf16_direct_rounding_brute_force():
    # Doubles that are not float32 values: a float32 detour could round twice.
    grid = _bf16_values_exact()
    rng = np.random.default_rng(11)
    xs = list(rng.standard_normal(300) * 10.0 ** rng.integers(-30, 30, 300))
    # Doubles just above a bfloat16 tie point (double rounding via f32 fails).
    xs += [1 + 2.0 ** -8 + 2.0 ** -40, 1 + 2.0 ** -8 - 2.0 ** -40]
    import bisect
    for x in xs:
        a = Fraction(abs(x))
        i = bisect.bisect_left(grid, a)
        lo = grid[max(i - 1, 0)] if i > 0 else grid[0]
        hi = grid[min(i, len(grid) - 1)]
        if a == hi:
            best = hi
        else:
            dlo, dhi = a - lo, hi - a
            if dlo < dhi:
                best = lo
            elif dhi < dlo:
                best = hi
            else:   # tie: even mantissa (low bit of the bfloat16 pattern)
                blo = grid.index(lo)
                best = lo if blo % 2 == 0 else hi
        got = numeric.bf16_bits_to_f64(numeric.f64_to_bf16_bits(np.array([x])))[0]
        assert Fraction(abs(got)) == best, x
        assert (got < 0) == (x < 0)


@pytest.mark.parametrize("x,expect", [
    (65504.0, 65504.0),
    (65519.99, 65504.0),
    (65520.0, np.inf),            # tie between 65504 and 2^16 goes to even -> inf
    (1 + 2.0 ** -11, 1.0),        # tie, even mantissa
    (1 + 3 * 2.0 ** -11, 1 + 2.0 ** -9),
    (2.0 ** -24, 2.0 ** -24),     # smallest subnormal
    (2.0 ** -25, 0.0),            # tie with zero -> even (zero)
])
def test_f16_rounding_special_values(x, expect):
    got = numeric.f16_bits_to_f64(numeric.f64_to_f16_bits(np.array([x])))[0]
    assert got == expect


def test_identity_conversion_keeps_nan_payload():
    bits = np.array([0x7FC1, 0xFFFF, 0x7F81, 0x1234], dtype=np.uint16)
    out = numeric.convert_bits(bits, "bf16", "bf16")
    np.testing.assert_array_equal(out, bits)


def test_widening_is_exact():
    rng = np.random.default_rng(3)
    b16 = rng.integers(0, 0x7F80, 5000, dtype=np.uint16)
    f32 = numeric.convert_bits(b16, "bf16", "f32")
    back = numeric.convert_bits(f32, "f32", "bf16")
    np.testing.assert_array_equal(back, b16)
