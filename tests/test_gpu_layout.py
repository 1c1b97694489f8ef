"""GPU parity of the Ulysses permutation kernels against the oracle (bit-exact).

Every buffer the CUDA path writes -- the peer-major send buffer, the received
blocks, the head layout and the sequence-sharded output -- is compared bit for
bit with the oracle's explicit index permutation.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import layout as olayout
from oracle import ulysses as ou
from tests.helpers import DT_NAME, bits

pytestmark = pytest.mark.gpu

CASES = [
    # B, S, H, D, U, R
    (1, 16, 4, 8, 2, 1),
    (1, 17, 5, 8, 3, 1),
    (2, 37, 5, 8, 3, 2),
    (1, 9, 3, 8, 4, 2),
    (1, 3, 2, 8, 2, 2),        # a rank with zero rows
    (2, 24, 24, 8, 5, 2),      # 24 heads over 5 ranks
    (1, 1000, 6, 128, 4, 2),   # several hundred rows per rank, D = 128
    (1, 257, 3, 64, 8, 1),
]


def _run_s2h(case, in_dt, wire_dt, dst_dts, nan_fill=False):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    planes = [synth.normal((B, S, H, D), 100 + p, 1.0, in_dt).cuda() for p in range(len(dst_dts))]
    send = torch.empty(L.wire_elems(len(planes)), dtype=synth.torch_dtype(wire_dt), device="cuda")
    recv = torch.empty_like(send)
    fill = float("nan") if nan_fill else 0.0
    heads = [torch.full(L.head_shape(), fill, dtype=synth.torch_dtype(dt), device="cuda") for dt in dst_dts]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, len(planes), send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, heads, flag)
    torch.cuda.synchronize()
    return L, planes, send, recv, heads, flag


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dts", [("bf16", "bf16", ("bf16", "bf16", "f16")),
                                 ("f32", "f32", ("f32", "f32", "f32")),
                                 ("f32", "bf16", ("bf16", "bf16", "bf16"))])
def test_s2h_bit_exact(case, dts):
    in_dt, wire_dt, dst_dts = dts
    L, planes, send, recv, heads, flag = _run_s2h(case, in_dt, wire_dt, dst_dts)
    ref = olayout.make_layout(*case)
    pb = [bits(p) for p in planes]
    o_send = ou.s2h_pack(ref, pb, in_dt, wire_dt)
    np.testing.assert_array_equal(bits(send), o_send)
    o_recv = ou.a2a(ref, "s2h", 3, o_send)
    np.testing.assert_array_equal(bits(recv), o_recv)
    ranks = ou.s2h_unpack(ref, o_recv, wire_dt, dst_dts)
    hb = [bits(h) for h in heads]
    for (r, v), pl in ranks.items():
        for p in range(3):
            got = hb[p][r, :, : ref.ring_len[r], v * ref.Hl:(v + 1) * ref.Hl]
            np.testing.assert_array_equal(got, pl[p])
    assert int(flag.item()) == 0


@pytest.mark.parametrize("case", CASES)
def test_h2s_bit_exact_and_roundtrip(case):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    ref = olayout.make_layout(*case)
    x = synth.normal((B, S, H, D), 7, 1.0, "bf16").cuda()
    send = torch.empty(L.wire_elems(1), dtype=torch.bfloat16, device="cuda")
    recv = torch.empty_like(send)
    head = torch.full(L.head_shape(), float("nan"), dtype=torch.bfloat16, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, [x], send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 1, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, [head])
    # head layout -> back, padded heads are NaN-free zeros, padded rows NaN
    send2 = torch.empty_like(send)
    recv2 = torch.empty_like(send)
    out = torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [head], send2)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, send2, recv2)
    sa.dit_ulysses_unpack(L, sa.DIT_HEAD_TO_SEQ, recv2, [out])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(out), bits(x))
    # against the oracle's head-to-seq wire
    hb = bits(head)
    o_ranks = {(r, v): hb[r, :, : ref.ring_len[r], v * ref.Hl:(v + 1) * ref.Hl]
               for r in range(R) for v in range(U)}
    o_send = ou.h2s_pack(ref, o_ranks, "bf16", "bf16")
    np.testing.assert_array_equal(bits(send2), o_send)
    np.testing.assert_array_equal(bits(recv2), ou.a2a(ref, "h2s", 1, o_send))


def test_h2s_output_cast_to_bf16_from_f32():
    import sequence_attention_gb300 as sa
    case = (2, 37, 5, 8, 3, 2)
    L = sa.dit_sp_layout_init(*case)
    ref = olayout.make_layout(*case)
    head = synth.normal(L.head_shape(), 3, 1.0, "f32").cuda()
    send = torch.empty(L.wire_elems(1), dtype=torch.float32, device="cuda")
    recv = torch.empty_like(send)
    out = torch.empty(L.seq_shape(), dtype=torch.bfloat16, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [head], send)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_HEAD_TO_SEQ, recv, [out])
    torch.cuda.synchronize()
    hb = bits(head)
    o_ranks = {(r, v): hb[r, :, : ref.ring_len[r], v * ref.Hl:(v + 1) * ref.Hl]
               for r in range(ref.R) for v in range(ref.U)}
    o_recv = ou.a2a(ref, "h2s", 1, ou.h2s_pack(ref, o_ranks, "f32", "f32"))
    np.testing.assert_array_equal(bits(out), ou.h2s_unpack(ref, o_recv, "f32", "bf16"))


def test_padding_rows_untouched_and_padded_heads_zero():
    case = (1, 37, 5, 8, 3, 2)     # ring blocks 19/18, heads 5 -> 6
    L, planes, send, recv, heads, flag = _run_s2h(case, "bf16", "bf16", ("bf16", "bf16", "bf16"),
                                                  nan_fill=True)
    h = heads[0].float().cpu()
    assert torch.isnan(h[1, :, 18:]).all()            # row past ring block 1's length
    assert (h[:, :, :, 5:][~torch.isnan(h[:, :, :, 5:])] == 0).all()
    assert not torch.isnan(h[0, :, :19, 5:]).any()    # padded head written as 0


def test_range_flag_on_f16_overflow():
    import sequence_attention_gb300 as sa
    case = (1, 16, 4, 8, 2, 1)
    L = sa.dit_sp_layout_init(*case)
    planes = [synth.normal((1, 16, 4, 8), 1 + p, 1.0, "bf16").cuda() for p in range(3)]
    planes[2][0, 3, 1, 2] = 1.0e6          # representable in bf16, not in f16
    send = torch.empty(L.wire_elems(3), dtype=torch.bfloat16, device="cuda")
    recv = torch.empty_like(send)
    heads = [torch.empty(L.head_shape(), dtype=dt, device="cuda")
             for dt in (torch.bfloat16, torch.bfloat16, torch.float16)]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 3, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, heads, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 5        # DIT_ERR_RANGE


@pytest.mark.parametrize("value,dst,flagged", [
    (65519.99609375, "f16", False),   # the largest float32 below the f16 midpoint: rounds to 65504
    (65520.0, "f16", True),           # the midpoint: the tie goes to the even neighbour, infinity
    (-65520.0, "f16", True),
    (float("inf"), "f16", False),     # already infinite: not a range error
    (float("nan"), "f16", False),
    (3.3961775e38, "bf16", True),     # (2 - 2^-8) * 2^127, the bf16 midpoint
    (3.3961773e38, "bf16", False),    # the float32 just below it
])
def test_range_flag_threshold(value, dst, flagged):
    """The range flag is raised exactly when round-to-nearest-even makes a
    finite value infinite (float32 wire, 16-bit destination)."""
    import sequence_attention_gb300 as sa
    L = sa.dit_sp_layout_init(1, 8, 2, 8, 2, 1)
    x = torch.ones((1, 8, 2, 8), dtype=torch.float32, device="cuda")
    x[0, 5, 1, 3] = value
    send = torch.empty(L.wire_elems(1), dtype=torch.float32, device="cuda")
    recv = torch.empty_like(send)
    out = [torch.empty(L.head_shape(), dtype=synth.torch_dtype(dst), device="cuda")]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, [x], send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 1, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, out, flag)
    torch.cuda.synchronize()
    assert (int(flag.item()) == 5) == flagged
    got = out[0][0, 0, 5, 1, 3].float().item()
    ref = torch.tensor([value], dtype=torch.float32).to(synth.torch_dtype(dst)).float().item()
    assert (got == ref) or (got != got and ref != ref)


@pytest.mark.parametrize("name,U", [("flux1024", 4), ("flux1008", 4), ("qwen1328", 5), ("wan", 8)])
def test_full_size_layout(name, U):
    """At the workloads' full sizes: S2H gives rank (r, v) exactly its slice of
    the global tensors (checked on the device for every rank), and H2S after
    S2H is the identity, bit for bit."""
    import sequence_attention_gb300 as sa
    w = synth.WORKLOADS[name]
    L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, U, w.R)
    q, k, v = w.qkv("cuda")
    send = torch.empty(L.wire_elems(3), dtype=torch.bfloat16, device="cuda")
    recv = torch.empty_like(send)
    heads = [torch.empty(L.head_shape(), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, [q, k, v], send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 3, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, heads)
    del send, recv
    for p, x in enumerate((q, k, v)):
        for r in range(L.R):
            rows = slice(L.ring_off[r], L.ring_off[r] + L.ring_len[r])
            got = heads[p][r, :, : L.ring_len[r], : w.H]
            assert torch.equal(got.view(torch.int16), x[:, rows].view(torch.int16))
        assert not heads[p][..., w.H:, :][:, :, : min(L.ring_len)].any()   # padded heads are 0
    out = torch.empty_like(q)
    s1 = torch.empty(L.wire_elems(1), dtype=torch.bfloat16, device="cuda")
    r1 = torch.empty_like(s1)
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [heads[1]], s1)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, s1, r1)
    sa.dit_ulysses_unpack(L, sa.DIT_HEAD_TO_SEQ, r1, [out])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), k.view(torch.int16))
