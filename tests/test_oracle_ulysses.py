"""Pins for the oracle's Ulysses all-to-all (an explicit permutation).

The head-sharded result is pinned to its meaning on the pages: after the
sequence-to-head exchange, rank (r, v) holds the full rows of ring block r
for the heads of group v (a plain slice of the global tensor), and the
head-to-sequence exchange gives every rank its own rows for all heads.  The
even case is also pinned to a textbook reshape/transpose of the send buffer.
"""
import numpy as np
import pytest

from oracle import layout, ulysses
from oracle.numeric import convert_bits


def _bits(shape, seed, dt="bf16"):
    rng = np.random.default_rng(seed)
    if dt == "f32":
        return rng.standard_normal(shape).astype(np.float32).view(np.uint32)
    return rng.integers(0, 0x7F80, size=shape, dtype=np.uint16)


CASES = [
    # B, S, H, D, U, R
    (1, 16, 4, 8, 2, 1),
    (1, 17, 5, 8, 3, 1),      # uneven rows, padded heads (5 -> 6)
    (2, 37, 5, 4, 3, 2),      # batch 2, USP 3x2, uneven everywhere
    (1, 9, 3, 8, 4, 2),       # ranks with 1 row
    (1, 3, 2, 4, 2, 2),       # a rank with zero rows
    (2, 24, 24, 4, 5, 2),     # 24 heads over 5 ranks (Qwen-like padding)
]


def _slice_with_padded_heads(x, rows, h0, Hl, H):
    B, _, _, D = x.shape
    out = np.zeros((B, len(range(*rows)), Hl, D), dtype=x.dtype)
    h1 = min(h0 + Hl, H)
    if h1 > h0:
        out[:, :, :h1 - h0] = x[:, rows[0]:rows[1], h0:h1]
    return out


# (pad_heads, pad_lcm64): padded heads (the default), padding-free uneven
# heads, and the lcm(SP, 64) sequence padding with either head layout
MODES = [(True, False), (False, False), (True, True), (False, True)]


def _slice_of(x, L, r, v):
    """Rows of ring block r (zero past S) and heads of group v (zero past H)
    of the global tensor x, as rank (r, v) must hold them."""
    B, S, H, D = x.shape
    out = np.zeros((B, L.ring_len[r], L.head_len[v], D), dtype=x.dtype)
    m = L.real_rows(r)
    h0, h1 = L.head_off[v], min(L.head_off[v] + L.head_len[v], H)
    if h1 > h0 and m > 0:
        out[:, :m, :h1 - h0] = x[:, L.ring_off[r]:L.ring_off[r] + m, h0:h1]
    return out


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("mode", MODES)
def test_s2h_gives_each_rank_its_heads_over_its_ring_block(case, mode):
    B, S, H, D, U, R = case
    L = layout.make_layout(B, S, H, D, U, R, pad_heads=mode[0], pad_lcm64=mode[1])
    planes = [_bits((B, S, H, D), 100 + p) for p in range(3)]
    send = ulysses.s2h_pack(L, planes, "bf16", "bf16")
    recv = ulysses.a2a(L, "s2h", 3, send)
    ranks = ulysses.s2h_unpack(L, recv, "bf16", ("bf16",) * 3)
    for r in range(R):
        for v in range(U):
            for p in range(3):
                np.testing.assert_array_equal(ranks[(r, v)][p], _slice_of(planes[p], L, r, v))
    if mode == (True, False):   # the original reading, written independently of the layout fields
        for r in range(R):
            rows = (L.ring_off[r], L.ring_off[r] + L.ring_len[r])
            for v in range(U):
                expect = _slice_with_padded_heads(planes[0], rows, v * L.Hl, L.Hl, H)
                np.testing.assert_array_equal(ranks[(r, v)][0], expect)


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("mode", MODES)
def test_h2s_after_s2h_is_identity(case, mode):
    B, S, H, D, U, R = case
    L = layout.make_layout(B, S, H, D, U, R, pad_heads=mode[0], pad_lcm64=mode[1])
    x = _bits((B, S, H, D), 7)
    x[0, 0, 0, 0] = 0x7FC1            # a NaN payload must survive untouched
    send = ulysses.s2h_pack(L, [x], "bf16", "bf16")
    ranks = ulysses.s2h_unpack(L, ulysses.a2a(L, "s2h", 1, send), "bf16", ("bf16",))
    o_ranks = {k: v[0] for k, v in ranks.items()}
    back = ulysses.h2s_unpack(L, ulysses.a2a(L, "h2s", 1,
                                             ulysses.h2s_pack(L, o_ranks, "bf16", "bf16")),
                              "bf16", "bf16")
    np.testing.assert_array_equal(back, x)


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("mode", MODES)
def test_padding_never_reaches_the_output(case, mode):
    B, S, H, D, U, R = case
    L = layout.make_layout(B, S, H, D, U, R, pad_heads=mode[0], pad_lcm64=mode[1])
    rng = np.random.default_rng(5)
    o_ranks = {}
    truth = np.zeros((B, S, H, D), dtype=np.uint16)
    for r in range(R):
        m = L.real_rows(r)
        for v in range(U):
            o = rng.integers(0, 0x7F80, size=(B, L.ring_len[r], L.head_len[v], D), dtype=np.uint16)
            h0, h1 = L.head_off[v], min(L.head_off[v] + L.head_len[v], H)
            o[:, :, max(h1 - h0, 0):] = 0x7FC0           # NaN in the padded heads
            o[:, m:] = 0x7FC0                             # and in the padding rows
            o_ranks[(r, v)] = o
            if h1 > h0:
                truth[:, L.ring_off[r]:L.ring_off[r] + m, h0:h1] = o[:, :m, :h1 - h0]
    send = ulysses.h2s_pack(L, o_ranks, "bf16", "bf16")
    out = ulysses.h2s_unpack(L, ulysses.a2a(L, "h2s", 1, send), "bf16", "bf16")
    np.testing.assert_array_equal(out, truth)
    assert not np.any(send == 0x7FC0)   # padding is zero on the wire, not NaN


def test_send_buffer_matches_textbook_reshape_when_even():
    # S % U == 0, H % U == 0, R = 1: rank u's send buffer is its rows,
    # reshaped [L, U, Hl, D] and transposed to peer-major [U, L, Hl, D].
    B, S, H, D, U = 1, 24, 6, 4, 3
    L = layout.make_layout(B, S, H, D, U, 1)
    x = _bits((B, S, H, D), 9)
    send = ulysses.s2h_pack(L, [x], "bf16", "bf16")
    Lr = S // U
    expect = np.concatenate([
        x[0, u * Lr:(u + 1) * Lr].reshape(Lr, U, H // U, D).transpose(1, 0, 2, 3).reshape(-1)
        for u in range(U)])
    np.testing.assert_array_equal(send, expect)
    # and rank v receives, in source order, those rows of its heads
    recv = ulysses.a2a(L, "s2h", 1, send)
    per = S * (H // U) * D
    for v in range(U):
        np.testing.assert_array_equal(
            recv[v * per:(v + 1) * per],
            x[0, :, v * (H // U):(v + 1) * (H // U)].reshape(-1))


def test_degree_one_is_identity():
    L = layout.make_layout(2, 11, 3, 4, 1, 1)
    x = _bits((2, 11, 3, 4), 10)
    send = ulysses.s2h_pack(L, [x], "bf16", "bf16")
    ranks = ulysses.s2h_unpack(L, ulysses.a2a(L, "s2h", 1, send), "bf16", ("bf16",))
    np.testing.assert_array_equal(ranks[(0, 0)][0], x)


def test_pack_cast_is_the_elementwise_cast_of_the_slice():
    # f32 inputs on a bf16 wire (the pages' optional F32->16-bit conversion);
    # V converted to f16 by the unpack.
    B, S, H, D, U, R = 1, 13, 3, 4, 2, 1
    L = layout.make_layout(B, S, H, D, U, R)
    planes = [_bits((B, S, H, D), 20 + p, "f32") for p in range(3)]
    send = ulysses.s2h_pack(L, planes, "f32", "bf16")
    ranks = ulysses.s2h_unpack(L, ulysses.a2a(L, "s2h", 3, send), "bf16",
                               ("bf16", "bf16", "f16"))
    for v in range(U):
        for p, dt in enumerate(("bf16", "bf16", "f16")):
            sl = _slice_with_padded_heads(planes[p], (0, S), v * L.Hl, L.Hl, H)
            expect = convert_bits(convert_bits(sl, "f32", "bf16"), "bf16", dt)
            np.testing.assert_array_equal(ranks[(0, v)][p], expect)
