"""GPU parity of the receive preparation with RoPE and of the paired
text/image stream path against the oracle.

The rotated Q/K planes are checked against the oracle's float64 rotation of
the received values within the fp32-then-round bound; every unrotated plane
and every joint-stream layout buffer is compared bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import layout as olayout
from oracle import rope as orope
from oracle import ulysses as ou
from tests.helpers import assert_rotation_close, bits, f64

pytestmark = pytest.mark.gpu

CASES = [
    # B, S, H, D, U, R
    (1, 16, 4, 8, 2, 1),
    (2, 37, 5, 8, 3, 2),
    (1, 3, 2, 8, 2, 2),        # a rank with zero rows
    (2, 24, 24, 16, 5, 2),     # 24 heads over 5 ranks: a padded head
    (1, 1000, 6, 128, 4, 2),   # several hundred rows per rank, D = 128
    (1, 257, 3, 64, 8, 1),
]

DTS = [("bf16", "bf16", ("bf16", "bf16", "f16")),
       ("f32", "f32", ("f32", "f32", "f32")),
       ("f32", "bf16", ("bf16", "bf16", "bf16")),
       ("bf16", "bf16", ("f32", "f32", "f32"))]   # widening: one destination size per call


def _exchange(sa, L, planes, wire_dt):
    send = torch.empty(L.wire_elems(len(planes)), dtype=synth.torch_dtype(wire_dt), device="cuda")
    recv = torch.empty_like(send)
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, len(planes), send, recv)
    return recv


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dts", DTS)
def test_receive_prep_rope(case, dts):
    import sequence_attention_gb300 as sa
    in_dt, wire_dt, dst_dts = dts
    B, S, H, D, U, R = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    ref = olayout.make_layout(*case)
    planes = [synth.normal((B, S, H, D), 300 + p, 1.0, in_dt).cuda() for p in range(3)]
    cos, sin = synth.rope_tables_linear(S, D)
    recv = _exchange(sa, L, planes, wire_dt)
    heads = [torch.full(L.head_shape(), float("nan"), dtype=synth.torch_dtype(dt), device="cuda")
             for dt in dst_dts]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_unpack_rope(L, recv, heads, cos.cuda(), sin.cuda(), 0b011, flag)
    torch.cuda.synchronize()
    want = orope.receive_prep(ref, bits(recv), wire_dt, list(dst_dts), cos.double().numpy(),
                              sin.double().numpy(), 0b011)
    xin = ou.s2h_unpack(ref, bits(recv), wire_dt, [wire_dt] * 3)
    from oracle import numeric
    for (r, v), pl in want.items():
        sl = (r, slice(None), slice(0, ref.ring_len[r]), slice(v * ref.Hl, (v + 1) * ref.Hl))
        for p in range(2):
            x = numeric.to_f64(xin[(r, v)][p], wire_dt)
            assert_rotation_close(f64(heads[p][sl]), pl[p], x, dst_dts[p], f"plane {p} rank ({r},{v})")
        np.testing.assert_array_equal(bits(heads[2][sl]), pl[2])
    assert int(flag.item()) == 0


@pytest.mark.parametrize("case", CASES[:4])
def test_zero_angles_and_empty_mask_equal_the_plain_unpack(case):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    planes = [synth.normal((B, S, H, D), 310 + p, 1.0, "bf16").cuda() for p in range(3)]
    recv = _exchange(sa, L, planes, "bf16")
    dts = (torch.bfloat16, torch.bfloat16, torch.float16)
    plain = [torch.zeros(L.head_shape(), dtype=t, device="cuda") for t in dts]
    zero = [torch.zeros(L.head_shape(), dtype=t, device="cuda") for t in dts]
    nomask = [torch.zeros(L.head_shape(), dtype=t, device="cuda") for t in dts]
    ones = torch.ones((S, D // 2), dtype=torch.float32, device="cuda")
    zeros = torch.zeros((S, D // 2), dtype=torch.float32, device="cuda")
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, plain)
    sa.dit_ulysses_unpack_rope(L, recv, zero, ones, zeros, 0b111)
    sa.dit_ulysses_unpack_rope(L, recv, nomask, ones * 0.5, zeros + 0.5, 0)
    torch.cuda.synchronize()
    for p in range(3):
        # cos 1, sin 0: x0*1 - x1*0 and x0*0 + x1*1 are exact in fp32
        assert torch.equal(zero[p], plain[p])
        np.testing.assert_array_equal(bits(nomask[p]), bits(plain[p]))


def test_rope_range_flag_on_f16_overflow():
    # a rotated bf16 value past the f16 range must set the flag
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = 1, 8, 2, 8, 2, 1
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    q = torch.full((B, S, H, D), 60000.0, dtype=torch.bfloat16, device="cuda")
    recv = _exchange(sa, L, [q], "bf16")
    out = [torch.zeros(L.head_shape(), dtype=torch.float16, device="cuda")]
    c = torch.full((S, D // 2), 0.70710678, dtype=torch.float32, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_unpack_rope(L, recv, out, c, c, 0b1, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == sa._lib.DIT_ERR_RANGE


def test_rope_argument_errors():
    import sequence_attention_gb300 as sa
    L = sa.dit_sp_layout_init(1, 8, 2, 8, 2, 1)
    recv = torch.zeros(L.wire_elems(1), dtype=torch.bfloat16, device="cuda")
    out = [torch.zeros(L.head_shape(), dtype=torch.bfloat16, device="cuda")]
    t = torch.ones((8, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(sa.DitError):
        sa.dit_ulysses_unpack_rope(L, recv, out, t, t, 0b10)     # plane 1 does not exist
    with pytest.raises(ValueError):
        sa.dit_ulysses_unpack_rope(L, recv, out, t[:7], t, 0b1)  # table too short


JOINT = [
    # B, S, H, D, U, R, S_txt
    (1, 16, 4, 8, 2, 1, 5),
    (2, 37, 5, 8, 3, 2, 12),    # the text/image boundary inside a rank
    (1, 9, 3, 8, 4, 2, 0),      # image only
    (1, 9, 3, 8, 4, 2, 9),      # text only
    (2, 24, 24, 16, 5, 2, 1),
    (1, 1000, 6, 128, 4, 2, 256),
]


def _split(t, s_txt):
    return t[:, :s_txt].contiguous(), t[:, s_txt:].contiguous()


@pytest.mark.parametrize("case", JOINT)
@pytest.mark.parametrize("dts", [("bf16", "bf16"), ("f32", "bf16"), ("f32", "f32")])
def test_joint_streams_bit_exact(case, dts):
    import sequence_attention_gb300 as sa
    in_dt, wire_dt = dts
    B, S, H, D, U, R, S_txt = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    ref = olayout.make_layout(B, S, H, D, U, R)
    joint = [synth.normal((B, S, H, D), 320 + p, 1.0, in_dt) for p in range(3)]
    txt = [_split(j, S_txt)[0].cuda() for j in joint] if S_txt > 0 else None
    img = [_split(j, S_txt)[1].cuda() for j in joint] if S_txt < S else None
    send = torch.empty(L.wire_elems(3), dtype=synth.torch_dtype(wire_dt), device="cuda")
    sa.dit_ulysses_pack_joint(L, txt, img, send)
    torch.cuda.synchronize()
    o_send = ou.s2h_pack(ref, [bits(j) for j in joint], in_dt, wire_dt)
    np.testing.assert_array_equal(bits(send), o_send)
    # the inverse: a head-layout tensor back into the two streams
    head = synth.normal(L.head_shape(), 330, 1.0, wire_dt).cuda()
    send_o = torch.empty(L.wire_elems(1), dtype=synth.torch_dtype(wire_dt), device="cuda")
    recv_o = torch.empty_like(send_o)
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [head], send_o)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, send_o, recv_o)
    out_t = torch.full((B, S_txt, H, D), float("nan"), dtype=torch.bfloat16, device="cuda") if S_txt else None
    out_i = torch.full((B, S - S_txt, H, D), float("nan"), dtype=torch.bfloat16, device="cuda") if S_txt < S else None
    sa.dit_ulysses_unpack_joint(L, recv_o, out_t, out_i)
    torch.cuda.synchronize()
    want = ou.h2s_unpack(ref, bits(recv_o), wire_dt, "bf16")
    if out_t is not None:
        np.testing.assert_array_equal(bits(out_t), want[:, :S_txt])
    if out_i is not None:
        np.testing.assert_array_equal(bits(out_i), want[:, S_txt:])


def test_joint_argument_errors():
    import sequence_attention_gb300 as sa
    L = sa.dit_sp_layout_init(1, 8, 2, 8, 2, 1)
    send = torch.zeros(L.wire_elems(1), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((1, 4, 2, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa.DitError):   # S_txt = 4 but no image stream
        sa.dit_ulysses_pack_joint(L, [x], None, send)
