"""USP composition (Ulysses inside, ring outside) equals plain attention.

The pages state the decomposition is exact (edge-dit.cpp "Parallel
execution"; SGLang Diffusion "Parallelism Overview"): every (U, R) split must
reproduce single-shot attention up to float64 summation order.
"""
import numpy as np
import pytest

from oracle import attention as att
from oracle import layout, usp


@pytest.mark.parametrize("B,S,H,D,U,R", [
    (1, 32, 4, 8, 2, 1),
    (1, 32, 4, 8, 1, 2),
    (1, 32, 4, 8, 2, 2),
    (2, 37, 5, 4, 3, 2),      # uneven rows and padded heads
    (1, 23, 3, 8, 2, 4),      # ring blocks of different length
    (1, 5, 2, 4, 4, 2),       # ranks with zero or one row
])
def test_usp_equals_single_shot(B, S, H, D, U, R):
    rng = np.random.default_rng(S * 131 + U * 7 + R)
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    L = layout.make_layout(B, S, H, D, U, R)
    o, lse_ranks = usp.usp_attention(L, q, k, v)
    o_ref, lse_ref = att.attention(q, k, v)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    for (r, vv), l in lse_ranks.items():
        h0, h1 = vv * L.Hl, min(vv * L.Hl + L.Hl, H)
        if h1 > h0:
            rows = slice(L.ring_off[r], L.ring_off[r] + L.ring_len[r])
            np.testing.assert_allclose(l[:, :h1 - h0], lse_ref[:, h0:h1, rows], atol=1e-13)


@pytest.mark.parametrize("pad_heads,pad_lcm64", [(False, False), (True, True), (False, True)])
@pytest.mark.parametrize("B,S,H,D,U,R", [(2, 37, 5, 4, 3, 2), (1, 23, 3, 8, 2, 4), (1, 130, 7, 4, 4, 1)])
def test_usp_equals_single_shot_in_every_layout(pad_heads, pad_lcm64, B, S, H, D, U, R):
    # no-pad uneven heads and lcm(SP, 64) sequence padding change only where
    # rows and heads travel; padding rows are no keys, so the result is the
    # same full attention
    rng = np.random.default_rng(S * 17 + U + 5 * R)
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    L = layout.make_layout(B, S, H, D, U, R, pad_heads=pad_heads, pad_lcm64=pad_lcm64)
    o, _ = usp.usp_attention(L, q, k, v)
    o_ref, _ = att.attention(q, k, v)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
