"""Pins for the oracle's rotary embedding: the properties that define it."""
import numpy as np
import pytest

from oracle import rope as orope


def _angles(S, D, base=10000.0, offset=0):
    i = np.arange(D // 2)
    theta = base ** (-2.0 * i / D)
    t = np.arange(S)[:, None] + offset
    return np.cos(t * theta), np.sin(t * theta), theta


def test_zero_angle_is_identity():
    x = np.random.default_rng(0).standard_normal((2, 5, 3, 8))
    y = orope.rope(x, np.ones((5, 4)), np.zeros((5, 4)))
    np.testing.assert_array_equal(y, x)


def test_pairs_keep_their_norm():
    x = np.random.default_rng(1).standard_normal((1, 7, 2, 16))
    c, s, _ = _angles(7, 16)
    y = orope.rope(x, c, s)
    n_x = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n_y = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(n_y, n_x, rtol=1e-13)


def test_inverse_rotation_restores_the_input():
    x = np.random.default_rng(2).standard_normal((1, 6, 2, 8))
    c, s, _ = _angles(6, 8)
    np.testing.assert_allclose(orope.rope(orope.rope(x, c, s), c, -s), x, atol=1e-13)


def test_quarter_turn_on_a_basis_vector():
    # angle pi/2 on pair 0 maps e0 -> e1 and e1 -> -e0 (a sign slip fails this)
    x = np.zeros((1, 2, 1, 4))
    x[0, 0, 0, 0] = 1.0
    x[0, 1, 0, 1] = 1.0
    c = np.array([[0.0, 1.0], [0.0, 1.0]])
    s = np.array([[1.0, 0.0], [1.0, 0.0]])
    y = orope.rope(x, c, s)
    np.testing.assert_allclose(y[0, 0, 0], [0, 1, 0, 0], atol=1e-15)
    np.testing.assert_allclose(y[0, 1, 0], [-1, 0, 0, 0], atol=1e-15)


def test_scores_depend_only_on_relative_position():
    # <R(m) q, R(n) k> is unchanged when both positions shift by the same amount
    rng = np.random.default_rng(3)
    D = 16
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    c, s, _ = _angles(40, D)
    xq = np.broadcast_to(q, (1, 40, 1, D)).copy()
    xk = np.broadcast_to(k, (1, 40, 1, D)).copy()
    rq, rk = orope.rope(xq, c, s)[0, :, 0], orope.rope(xk, c, s)[0, :, 0]
    d1 = rq[5] @ rk[2]
    d2 = rq[25] @ rk[22]
    d3 = rq[30] @ rk[27]
    np.testing.assert_allclose([d2, d3], [d1, d1], rtol=1e-12)
    assert abs(rq[5] @ rk[2] - rq[5] @ rk[3]) > 1e-6


def test_joint_sequence_puts_text_first():
    t = np.full((1, 2, 1, 1), 1.0)
    i = np.full((1, 3, 1, 1), 2.0)
    np.testing.assert_array_equal(orope.joint(t, i)[0, :, 0, 0], [1, 1, 2, 2, 2])


def _global_planes(B, S, H, D, n, dt, seed):
    import synth
    from tests.helpers import bits
    ts = [synth.normal((B, S, H, D), seed + p, 1.0, dt) for p in range(n)]
    return [bits(t) for t in ts]


@pytest.mark.parametrize("pad_lcm64", [False, True])
def test_receive_prep_matches_direct_indexing(pad_lcm64):
    # brute force: every head-layout element of every rank, read straight
    # from the rotated global planes (no send/receive bookkeeping); rows of
    # the padded layout at or past S are zero and unrotated
    import synth
    from oracle import layout as olayout, numeric, ulysses
    B, S, H, D, U, R = 2, 23, 5, 8, 3, 2
    L = olayout.make_layout(B, S, H, D, U, R, pad_lcm64=pad_lcm64)
    planes = _global_planes(B, S, H, D, 3, "bf16", 40)
    cos, sin = (t.numpy().astype(np.float64) for t in synth.rope_tables_linear(S, D))
    recv = ulysses.a2a(L, "s2h", 3, ulysses.s2h_pack(L, planes, "bf16", "bf16"))
    got = orope.receive_prep(L, recv, "bf16", ["bf16", "bf16", "f16"], cos, sin, 0b011)
    rotated = [orope.rope(numeric.to_f64(planes[p], "bf16"), cos, sin) for p in range(2)]
    for (r, v), pl in got.items():
        for s in range(L.ring_len[r]):
            t = L.ring_off[r] + s
            for hl in range(L.Hl):
                h = v * L.Hl + hl
                real = h < H and t < S
                for p in range(2):
                    want = rotated[p][:, t, h] if real else np.zeros((B, D))
                    np.testing.assert_array_equal(pl[p][:, s, hl], want)
                want_v = (numeric.convert_bits(planes[2][:, t, h], "bf16", "f16") if real
                          else np.zeros((B, D), np.uint16))
                np.testing.assert_array_equal(pl[2][:, s, hl], want_v)
    assert (L.S_pad > S) == pad_lcm64


def test_receive_prep_with_zero_angles_is_the_plain_unpack():
    from oracle import layout as olayout, numeric, ulysses
    B, S, H, D, U, R = 1, 11, 4, 8, 2, 1
    L = olayout.make_layout(B, S, H, D, U, R)
    planes = _global_planes(B, S, H, D, 2, "f32", 50)
    recv = ulysses.a2a(L, "s2h", 2, ulysses.s2h_pack(L, planes, "f32", "f32"))
    got = orope.receive_prep(L, recv, "f32", ["f32", "f32"], np.ones((S, 4)), np.zeros((S, 4)), 0b11)
    plain = ulysses.s2h_unpack(L, recv, "f32", ["f32", "f32"])
    for key, pl in got.items():
        for p in range(2):
            np.testing.assert_array_equal(pl[p], numeric.to_f64(plain[key][p], "f32"))
