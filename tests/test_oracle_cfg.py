"""Pins for the oracle's classifier-free guidance combine."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import cfg
from oracle.numeric import bf16_bits_to_f64, f64_to_bf16_bits


def _bf16_pair(n, seed):
    rng = np.random.default_rng(seed)
    t = torch.from_numpy(rng.standard_normal((2, n)).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_g0_is_uncond_bit_exact():
    p = _bf16_pair(4096, 1)
    np.testing.assert_array_equal(cfg.cfg_combine_bits(p, "bf16", 0.0, "bf16"), p[0])


def test_g1_is_cond_bit_exact():
    p = _bf16_pair(4096, 2)
    np.testing.assert_array_equal(cfg.cfg_combine_bits(p, "bf16", 1.0, "bf16"), p[1])


def test_equal_branches_are_fixed_points():
    p = _bf16_pair(1024, 3)
    p[1] = p[0]
    for g in (0.5, 3.5, 7.0, -2.0):
        np.testing.assert_array_equal(cfg.cfg_combine_bits(p, "bf16", g, "bf16"), p[0])


def test_linear_in_g():
    rng = np.random.default_rng(4)
    u, c = rng.standard_normal(100), rng.standard_normal(100)
    d1 = cfg.cfg_combine_f64(u, c, 1.5) - u
    d2 = cfg.cfg_combine_f64(u, c, 2.0) - u
    d3 = cfg.cfg_combine_f64(u, c, 3.5) - u
    np.testing.assert_allclose(d3, d1 + d2, atol=1e-13)


@pytest.mark.parametrize("g", [3.5, 4.0, 5.0])
def test_brute_force_exact_rational(g):
    # Exact rational u + g(c - u), then nearest bfloat16 by scanning the grid
    # around it: independent of the oracle's float64 evaluation and rounding.
    p = _bf16_pair(64, 5)
    got = bf16_bits_to_f64(cfg.cfg_combine_bits(p, "bf16", g, "bf16"))
    u, c = bf16_bits_to_f64(p[0]), bf16_bits_to_f64(p[1])
    for i in range(64):
        exact = Fraction(u[i]) + Fraction(g) * (Fraction(c[i]) - Fraction(u[i]))
        guess = bf16_bits_to_f64(f64_to_bf16_bits(np.array([float(exact)])))[0]
        # candidates: the three neighbours of the guess on the bfloat16 grid
        b = int(f64_to_bf16_bits(np.array([guess]))[0])
        cands = [bf16_bits_to_f64(np.array([x], dtype=np.uint16))[0]
                 for x in (b - 1, b, b + 1) if 0 <= x < 0x10000]
        best = min(cands, key=lambda y: (abs(Fraction(y) - exact),
                                         int(f64_to_bf16_bits(np.array([y]))[0]) & 1))
        assert got[i] == best
