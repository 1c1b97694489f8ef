"""Pins for the oracle's sequence split, head padding and a2a bookkeeping."""
import json
import os

import pytest

from oracle import layout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("S,n,lens", [
    # Workload splits, worked by hand from "first S mod n ranks get +1":
    (4481, 2, [2241, 2240]),            # 4481 = 2*2240 + 1
    (2241, 4, [561, 560, 560, 560]),    # 2241 = 4*560 + 1
    (2240, 4, [560, 560, 560, 560]),
    (7145, 2, [3573, 3572]),            # 7145 = 2*3572 + 1
    (3573, 5, [715, 715, 715, 714, 714]),   # 3573 = 5*714 + 3
    (3572, 5, [715, 715, 714, 714, 714]),   # 3572 = 5*714 + 2
    (75600, 4, [18900] * 4),
    (18900, 8, [2363] * 4 + [2362] * 4),    # 18900 = 8*2362 + 4
    (4608, 4, [1152] * 4),
    (3, 5, [1, 1, 1, 0, 0]),
    (0, 3, [0, 0, 0]),
])
def test_balanced_split(S, n, lens):
    got, offs = layout.balanced_split(S, n)
    assert got == lens
    assert offs == [sum(lens[:i]) for i in range(n)]


def test_balanced_split_properties():
    for S in range(0, 60):
        for n in range(1, 9):
            lens, offs = layout.balanced_split(S, n)
            assert sum(lens) == S
            assert max(lens) - min(lens) <= 1
            assert lens == sorted(lens, reverse=True)


def test_golden_shape_statements():
    """Shape chains and head examples stated on the pages (see the fixture)."""
    with open(os.path.join(GOLDEN, "shape_statements.json")) as f:
        g = json.load(f)
    for case in g["ulysses_shapes"]:
        B, S, H, D, P = (case[x] for x in ("B", "S", "H", "D", "P"))
        L = layout.make_layout(B, S, H, D, P, 1)
        # seq-sharded [B, S/P, H, D] per rank -> head-sharded [B, S, H/P, D]
        assert all(n == case["local_S"] for n in L.rank_len)
        assert L.S_cap == case["full_S"] and L.Hl == case["local_H"]
    for case in g["usp_shapes"]:
        B, S, H, D, U, R = (case[x] for x in ("B", "S", "H", "D", "U", "R"))
        L = layout.make_layout(B, S, H, D, U, R)
        assert all(n == case["S_over_UR"] for n in L.rank_len)
        assert all(n == case["S_over_R"] for n in L.ring_len)
        assert L.Hl == case["H_over_U"]
    for case in g["head_divisibility"]:
        Hp, Hl = layout.padded_heads(case["local_heads"], case["U"])
        assert (Hp == case["local_heads"]) == case["divisible"]
        assert Hp % case["U"] == 0 and Hp - case["local_heads"] < case["U"]


@pytest.mark.parametrize("H,U,Hp,Hl", [(24, 5, 25, 5), (24, 4, 24, 6), (30, 4, 32, 8),
                                       (40, 8, 40, 5), (1, 3, 3, 1), (24, 2, 24, 12)])
def test_padded_heads(H, U, Hp, Hl):
    assert layout.padded_heads(H, U) == (Hp, Hl)


def test_rank_order_partitions_the_sequence():
    L = layout.make_layout(2, 7145, 24, 128, 5, 2)
    acc = 0
    for rid in range(L.R * L.U):
        assert L.rank_off[rid] == acc
        acc += L.rank_len[rid]
    assert acc == L.S
    assert L.ring_len == (3573, 3572) and L.ring_off == (0, 3573)


@pytest.mark.parametrize("direction", ["s2h", "h2s"])
@pytest.mark.parametrize("dims", [(2, 7145, 24, 8, 5, 2), (1, 37, 5, 4, 3, 2), (1, 4481, 24, 8, 4, 2)])
def test_counts_are_consistent(direction, dims):
    B, S, H, D, U, R = dims
    L = layout.make_layout(B, S, H, D, U, R)
    nplanes = 3 if direction == "s2h" else 1
    for r in range(R):
        for u in range(U):
            sc, sd, _, _ = layout.a2a_counts(L, direction, nplanes, L.rank(r, u))
            for v in range(U):
                _, _, rc, rd = layout.a2a_counts(L, direction, nplanes, L.rank(r, v))
                assert sc[v] == rc[u]          # what u sends v is what v gets from u
            assert sd == [sum(sc[:i]) for i in range(U)]
    send_base, recv_base, total = layout.buffer_bases(L, direction, nplanes)
    assert total == nplanes * B * S * L.Hp * D


@pytest.mark.parametrize("S,sp,S_pad", [(4608, 4, 4608), (4481, 8, 4544), (7145, 10, 7360),
                                        (75600, 32, 75648), (0, 4, 0), (1, 3, 192), (191, 3, 192)])
def test_padded_length_is_the_next_multiple_of_lcm_sp_64(S, sp, S_pad):
    # hand-worked: lcm(8, 64) = 64, lcm(10, 64) = 320, lcm(3, 64) = 192
    assert layout.padded_length(S, sp) == S_pad


@pytest.mark.parametrize("H,U,lens", [(24, 5, [5, 5, 5, 5, 4]), (30, 4, [8, 8, 7, 7]),
                                      (40, 8, [5] * 8), (2, 3, [1, 1, 0])])
def test_unpadded_heads_are_split_without_padding(H, U, lens):
    L = layout.make_layout(1, 10, H, 8, U, 1, pad_heads=False)
    assert list(L.head_len) == lens and L.Hp == H and L.Hl == max(lens)
    assert list(L.head_off) == [sum(lens[:v]) for v in range(U)]


def test_lcm_padding_splits_the_padded_length_evenly():
    L = layout.make_layout(1, 4481, 24, 8, 4, 2, pad_lcm64=True)
    assert L.S == 4481 and L.S_pad == 4544
    assert set(L.rank_len) == {568} and L.ring_len == (2272, 2272)
    assert [L.real_rows(r) for r in range(2)] == [2272, 2209]


@pytest.mark.parametrize("direction", ["s2h", "h2s"])
@pytest.mark.parametrize("flags", [(False, False), (False, True), (True, True)])
@pytest.mark.parametrize("dims", [(2, 717, 24, 8, 5, 2), (1, 37, 5, 4, 3, 2)])
def test_counts_are_consistent_in_every_layout(direction, flags, dims):
    B, S, H, D, U, R = dims
    L = layout.make_layout(B, S, H, D, U, R, pad_heads=flags[0], pad_lcm64=flags[1])
    nplanes = 3 if direction == "s2h" else 1
    for r in range(R):
        for u in range(U):
            sc, sd, _, _ = layout.a2a_counts(L, direction, nplanes, L.rank(r, u))
            for v in range(U):
                _, _, rc, rd = layout.a2a_counts(L, direction, nplanes, L.rank(r, v))
                assert sc[v] == rc[u]
    _, _, total = layout.buffer_bases(L, direction, nplanes)
    assert total == nplanes * B * L.S_pad * L.Hp * D
