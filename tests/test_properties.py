"""Property-based pins over random sizes (hypothesis; skipped where it is not
installed): the C layout equals the oracle's for every size and flag, the
oracle's exchange is a bijection (seq->head then head->seq is the identity)
in every layout mode, and the e4m3 encoder agrees with PyTorch's cast."""
import ctypes

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import fp8 as ofp8  # noqa: E402
from oracle import layout as olayout  # noqa: E402
from oracle import ulysses as ou  # noqa: E402

sizes = st.tuples(st.integers(1, 3), st.integers(0, 300), st.integers(1, 48), st.sampled_from([8, 16, 64, 128]),
                  st.integers(1, 8), st.integers(1, 8))
flags = st.tuples(st.booleans(), st.booleans())


@settings(max_examples=300, deadline=None)
@given(sizes, flags)
def test_c_layout_equals_the_oracle(dims, fl):
    from sequence_attention_gb300 import _lib
    B, S, H, D, U, R = dims
    lay = _lib.DitSpLayout()
    f = (0 if fl[0] else _lib.DIT_LAYOUT_NOPAD_HEADS) | (_lib.DIT_LAYOUT_PAD_LCM64 if fl[1] else 0)
    assert _lib.lib().dit_sp_layout_init_ex(B, S, H, D, U, R, f, ctypes.byref(lay)) == 0
    ref = olayout.make_layout(B, S, H, D, U, R, pad_heads=fl[0], pad_lcm64=fl[1])
    assert (lay.Hp, lay.Hl, lay.S_cap, lay.S_pad) == (ref.Hp, ref.Hl, ref.S_cap, ref.S_pad)
    assert list(lay.head_len)[:U] == list(ref.head_len) and list(lay.head_off)[:U] == list(ref.head_off)
    assert list(lay.ring_len)[:R] == list(ref.ring_len)
    assert list(lay.rank_len)[:U * R] == list(ref.rank_len) and list(lay.rank_off)[:U * R] == list(ref.rank_off)
    for d, name in ((0, "s2h"), (1, "h2s")):
        rank = (S * 7 + U) % (U * R)
        arrs = [(ctypes.c_int64 * U)() for _ in range(4)]
        assert _lib.lib().dit_sp_a2a_counts(ctypes.byref(lay), d, 1, rank, *arrs) == 0
        exp = olayout.a2a_counts(ref, name, 1, rank)
        assert [list(a) for a in arrs] == [list(e) for e in exp]


@settings(max_examples=150, deadline=None)
@given(st.tuples(st.integers(1, 2), st.integers(0, 70), st.integers(1, 9), st.sampled_from([4, 8]),
                 st.integers(1, 5), st.integers(1, 3)), flags, st.integers(0, 2 ** 31))
def test_exchange_round_trip_is_the_identity(dims, fl, seed):
    B, S, H, D, U, R = dims
    L = olayout.make_layout(B, S, H, D, U, R, pad_heads=fl[0], pad_lcm64=fl[1])
    x = np.random.default_rng(seed).integers(0, 0x7F80, size=(B, S, H, D), dtype=np.uint16)
    ranks = ou.s2h_unpack(L, ou.a2a(L, "s2h", 1, ou.s2h_pack(L, [x], "bf16", "bf16")), "bf16", ("bf16",))
    o_ranks = {k: v[0] for k, v in ranks.items()}
    back = ou.h2s_unpack(L, ou.a2a(L, "h2s", 1, ou.h2s_pack(L, o_ranks, "bf16", "bf16")), "bf16", "bf16")
    np.testing.assert_array_equal(back, x)


@settings(max_examples=200, deadline=None)
@given(st.lists(st.floats(min_value=-460.0, max_value=460.0, width=32), min_size=1, max_size=64))
def test_e4m3_encoding_agrees_with_torch(vals):
    import torch
    y = np.asarray(vals, dtype=np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ofp8.e4m3_encode(y), ref)
