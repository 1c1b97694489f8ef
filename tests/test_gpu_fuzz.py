"""Seeded random layouts through the GPU permutation kernels, bit for bit
against the oracle: Ulysses degrees up to 8, ring degrees up to 4, either
layout flag, head counts below the degree (empty head groups without
padding), sequence lengths from 0 up, batches up to 3, the 16-bit and the
e4m3 wire, both directions."""
import numpy as np
import pytest
import torch

from oracle import fp8 as ofp8
from oracle import layout as olayout
from oracle import ulysses as ou
from tests.helpers import bits

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    U = int(rng.integers(1, 9))
    R = int(rng.integers(1, 5))
    return (int(rng.integers(1, 4)), int(rng.integers(0, 200)), int(rng.integers(1, 13)),
            int(rng.choice([16, 32, 64])), U, R, bool(rng.integers(0, 2)), bool(rng.integers(0, 2)))


# the largest rank counts the layout takes (DIT_MAX_RANKS = 64 virtual
# ranks, DIT_MAX_R = 8 ring blocks), with uneven rows and head groups
MAX_CASES = [(1, 701, 5, 16, 64, 1, True, False), (2, 301, 3, 32, 8, 8, False, True),
             (1, 517, 70, 16, 64, 1, False, False), (1, 129, 9, 64, 2, 8, True, True)]
# an empty sequence (every buffer has zero bytes, so its pointer is NULL),
# with and without the lcm(U*R, 64) padding; the first is the draw of seed 432
EMPTY_CASES = [(3, 0, 9, 32, 1, 4, True, True), (1, 0, 5, 64, 4, 2, False, False)]


@pytest.mark.parametrize("seed", list(range(40)) + [f"max{i}" for i in range(len(MAX_CASES))]
                         + [f"empty{i}" for i in range(len(EMPTY_CASES))])
def test_random_layouts_bit_exact(seed):
    import sequence_attention_gb300 as sa
    if isinstance(seed, str) and seed.startswith("max"):
        B, S, H, D, U, R, ph, pl = MAX_CASES[int(seed[3:])]
        seed = 500 + int(seed[3:])
    elif isinstance(seed, str):
        B, S, H, D, U, R, ph, pl = EMPTY_CASES[int(seed[5:])]
        seed = 600 + int(seed[5:])
    else:
        B, S, H, D, U, R, ph, pl = _case(seed)
    L = sa.dit_sp_layout_init(B, S, H, D, U, R, pad_heads=ph, pad_lcm64=pl)
    ref = olayout.make_layout(B, S, H, D, U, R, pad_heads=ph, pad_lcm64=pl)
    rng = np.random.default_rng(seed)
    planes = [torch.from_numpy(rng.integers(0, 0x7F80, size=(B, S, H, D), dtype=np.uint16).view(np.int16))
              .view(torch.bfloat16).cuda() for _ in range(2)]
    # 16-bit wire, seq -> head and back
    send = torch.empty(max(L.wire_elems(2), 1), dtype=torch.bfloat16, device="cuda")
    recv = torch.empty_like(send)
    heads = [torch.full(L.head_shape(), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 2, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, heads)
    out = torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    s1 = torch.empty(max(L.wire_elems(1), 1), dtype=torch.bfloat16, device="cuda")
    r1 = torch.empty_like(s1)
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [heads[0]], s1)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, s1, r1)
    sa.dit_ulysses_unpack(L, sa.DIT_HEAD_TO_SEQ, r1, [out])
    torch.cuda.synchronize()
    pb = [bits(p) for p in planes]
    o_send = ou.s2h_pack(ref, pb, "bf16", "bf16")
    n = o_send.size
    np.testing.assert_array_equal(bits(send)[:n], o_send)
    o_recv = ou.a2a(ref, "s2h", 2, o_send)
    np.testing.assert_array_equal(bits(recv)[:n], o_recv)
    for (r, v), pls in ou.s2h_unpack(ref, o_recv, "bf16", ("bf16", "bf16")).items():
        for p in range(2):
            got = bits(heads[p])[r, :, : ref.ring_len[r], ref.head_off[v]:ref.head_off[v] + ref.head_len[v]]
            np.testing.assert_array_equal(got, pls[p])
    np.testing.assert_array_equal(bits(out), pb[0])
    # e4m3 wire, seq -> head
    s8 = torch.empty(max(L.wire_bytes_e4m3(2), 16), dtype=torch.uint8, device="cuda")
    r8 = torch.empty_like(s8)
    h8 = [torch.full(L.head_shape(), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, s8)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 2, s8, r8)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, r8, h8)
    torch.cuda.synchronize()
    o8 = ofp8.s2h_pack(ref, pb, "bf16")
    n8 = o8.size * 2
    np.testing.assert_array_equal(s8.cpu().numpy()[:n8], o8.view(np.uint8))
    for (r, v), pls in ofp8.s2h_unpack(ref, ofp8.a2a(ref, "s2h", 2, o8), ["bf16", "bf16"]).items():
        for p in range(2):
            got = bits(h8[p])[r, :, : ref.ring_len[r], ref.head_off[v]:ref.head_off[v] + ref.head_len[v]]
            np.testing.assert_array_equal(got, pls[p])
