"""GPU parity of the e4m3 wire (Q, V and O in float8 with one scale per
(token, head); K stays 16-bit) against the oracle.

Every code is decided by IEEE float32 operations on both sides, so the send
buffers, the exchanged records and the decoded planes are compared bit for
bit.  End to end, attention over the decoded Q and V meets the bf16 bars
against the oracle's attention over the same decoded values; with O also
on the e4m3 wire the bound is derived from the format (see the test).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import fp8 as ofp8
from oracle import layout as olayout
from oracle import numeric
from oracle import rope as orope
from tests.helpers import assert_bf16_close, assert_rotation_close, bits, f64, rel_rms

pytestmark = pytest.mark.gpu

CASES = [
    # B, S, H, D, U, R
    (1, 16, 4, 16, 2, 1),
    (2, 37, 5, 32, 3, 2),
    (1, 3, 2, 16, 2, 2),       # a rank with zero rows
    (2, 24, 24, 64, 5, 2),     # 24 heads over 5 ranks: a padded head
    (1, 1000, 6, 128, 4, 2),   # several hundred rows per rank, D = 128
    (1, 77, 3, 256, 2, 1),     # 32 lanes per head
]


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def _s2h(sa, case, in_dt, dst_dts, seed=400):
    B, S, H, D, U, R = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    planes = [synth.normal((B, S, H, D), seed + p, 1.0, in_dt).cuda() for p in range(len(dst_dts))]
    send = torch.empty(L.wire_bytes_e4m3(len(planes)), dtype=torch.uint8, device="cuda")
    recv = torch.empty_like(send)
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, len(planes), send, recv)
    return L, planes, send, recv


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dts", [("bf16", ("bf16", "f16")), ("f32", ("f32", "f32")), ("bf16", ("f32", "f32"))])
def test_s2h_e4m3_bit_exact(case, dts):
    import sequence_attention_gb300 as sa
    in_dt, dst_dts = dts
    L, planes, send, recv = _s2h(sa, case, in_dt, dst_dts)
    heads = [torch.full(L.head_shape(), float("nan"), dtype=synth.torch_dtype(dt), device="cuda")
             for dt in dst_dts]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, heads, flag)
    torch.cuda.synchronize()
    ref = olayout.make_layout(*case)
    o_send = ofp8.s2h_pack(ref, [bits(p) for p in planes], in_dt)
    np.testing.assert_array_equal(_bytes(send), o_send.view(np.uint8))
    o_recv = ofp8.a2a(ref, "s2h", len(planes), o_send)
    np.testing.assert_array_equal(_bytes(recv), o_recv.view(np.uint8))
    for (r, v), pl in ofp8.s2h_unpack(ref, o_recv, list(dst_dts)).items():
        for p in range(len(dst_dts)):
            got = bits(heads[p])[r, :, : ref.ring_len[r], v * ref.Hl:(v + 1) * ref.Hl]
            np.testing.assert_array_equal(got, pl[p])
    assert int(flag.item()) == 0


@pytest.mark.parametrize("case", CASES)
def test_h2s_e4m3_bit_exact(case):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    ref = olayout.make_layout(*case)
    head = synth.normal(L.head_shape(), 410, 1.0, "bf16").cuda()
    send = torch.empty(L.wire_bytes_e4m3(1), dtype=torch.uint8, device="cuda")
    recv = torch.empty_like(send)
    out = torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [head], send)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_HEAD_TO_SEQ, recv, [out])
    torch.cuda.synchronize()
    hb = bits(head)
    o_ranks = {(r, v): hb[r, :, : ref.ring_len[r], v * ref.Hl:(v + 1) * ref.Hl]
               for r in range(R) for v in range(U)}
    o_send = ofp8.h2s_pack(ref, o_ranks, "bf16")
    np.testing.assert_array_equal(_bytes(send), o_send.view(np.uint8))
    o_recv = ofp8.a2a(ref, "h2s", 1, o_send)
    np.testing.assert_array_equal(_bytes(recv), o_recv.view(np.uint8))
    np.testing.assert_array_equal(bits(out), ofp8.h2s_unpack(ref, o_recv, "bf16"))


@pytest.mark.parametrize("case", [(2, 37, 5, 32, 3, 2, 12), (1, 1000, 6, 128, 4, 2, 256)])
def test_joint_streams_e4m3(case):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R, S_txt = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    ref = olayout.make_layout(B, S, H, D, U, R)
    joint = [synth.normal((B, S, H, D), 420 + p, 1.0, "bf16") for p in range(2)]
    txt = [j[:, :S_txt].contiguous().cuda() for j in joint]
    img = [j[:, S_txt:].contiguous().cuda() for j in joint]
    send = torch.empty(L.wire_bytes_e4m3(2), dtype=torch.uint8, device="cuda")
    sa.dit_ulysses_pack_joint(L, txt, img, send)
    head = synth.normal(L.head_shape(), 430, 1.0, "f32").cuda()
    send_o = torch.empty(L.wire_bytes_e4m3(1), dtype=torch.uint8, device="cuda")
    recv_o = torch.empty_like(send_o)
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [head], send_o)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, send_o, recv_o)
    out_t = torch.empty((B, S_txt, H, D), dtype=torch.bfloat16, device="cuda")
    out_i = torch.empty((B, S - S_txt, H, D), dtype=torch.bfloat16, device="cuda")
    sa.dit_ulysses_unpack_joint(L, recv_o, out_t, out_i)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bytes(send), ofp8.s2h_pack(ref, [bits(j) for j in joint], "bf16").view(np.uint8))
    want = ofp8.h2s_unpack(ref, _bytes(recv_o).view(np.uint16), "bf16")
    np.testing.assert_array_equal(bits(out_t), want[:, :S_txt])
    np.testing.assert_array_equal(bits(out_i), want[:, S_txt:])


@pytest.mark.parametrize("case", CASES[1:5])
def test_receive_prep_e4m3_rope(case):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L, planes, send, recv = _s2h(sa, case, "bf16", ("bf16", "f16"), seed=440)
    cos, sin = synth.rope_tables_linear(S, D)
    heads = [torch.zeros(L.head_shape(), dtype=torch.bfloat16, device="cuda"),
             torch.zeros(L.head_shape(), dtype=torch.float16, device="cuda")]
    sa.dit_ulysses_unpack_rope(L, recv, heads, cos.cuda(), sin.cuda(), 0b01)
    torch.cuda.synchronize()
    ref = olayout.make_layout(*case)
    dec = ofp8.s2h_unpack(ref, _bytes(recv).view(np.uint16), ["f32", "f16"])
    c, s = cos.double().numpy(), sin.double().numpy()
    for (r, v), pl in dec.items():
        sl = (r, slice(None), slice(0, ref.ring_len[r]), slice(v * ref.Hl, (v + 1) * ref.Hl))
        x = numeric.to_f64(pl[0], "f32")
        rows = slice(ref.ring_off[r], ref.ring_off[r] + ref.ring_len[r])
        want = orope.rope(x, c[rows], s[rows])
        assert_rotation_close(f64(heads[0][sl]), want, x, "bf16", f"Q rank ({r},{v})")
        np.testing.assert_array_equal(bits(heads[1][sl]), pl[1])


def test_e4m3_range_flag_and_errors():
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = 1, 8, 2, 16, 2, 1
    L = sa.dit_sp_layout_init(B, S, H, D, U, R)
    x = torch.full((B, S, H, D), 1.0e5, dtype=torch.bfloat16, device="cuda")
    send = torch.empty(L.wire_bytes_e4m3(1), dtype=torch.uint8, device="cuda")
    recv = torch.empty_like(send)
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, [x], send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 1, send, recv)
    out = [torch.zeros(L.head_shape(), dtype=torch.float16, device="cuda")]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, out, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == sa._lib.DIT_ERR_RANGE
    L24 = sa.dit_sp_layout_init(1, 8, 2, 24, 2, 1)          # D = 24 has no e4m3 wire
    y = torch.zeros((1, 8, 2, 24), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa.DitError):
        sa.dit_ulysses_pack(L24, sa.DIT_SEQ_TO_HEAD, [y], torch.empty(4096, dtype=torch.uint8, device="cuda"))
    with pytest.raises(sa.DitError):   # e4m3 is a wire type, not an element type
        sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, [send.view(1, -1)], recv)


def test_checked_exchange_carries_records():
    import sequence_attention_gb300 as sa
    case = (1, 1000, 6, 128, 4, 2)
    L, planes, send, recv = _s2h(sa, case, "bf16", ("bf16", "f16"))
    recv2 = torch.zeros_like(recv)
    arrival = torch.zeros(8, dtype=torch.int32, device="cuda")   # U * R counters
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_sp_signal(L, arrival, 1)
    sa.dit_a2a_sim_checked(L, sa.DIT_SEQ_TO_HEAD, 2, send, recv2, arrival, 1, 10 ** 9, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(recv, recv2)


def _usp_inputs(B, S, H, D, seed):
    return [synth.normal((B, S, H, D), seed + p, 0.5, "bf16") for p in range(3)]


def _decoded(x):
    """The oracle's e4m3 round trip of every (token, head) of x [B,S,H,D]."""
    return ofp8.dequantize_heads(*ofp8.quantize_heads(f64(x).astype(np.float32))).astype(np.float64)


@pytest.mark.parametrize("B,S,H,U,R", [(1, 700, 5, 2, 2), (2, 517, 4, 3, 1)])
def test_usp_e4m3_qv_meets_bf16_bars_on_decoded_inputs(B, S, H, U, R):
    from sequence_attention_gb300.usp import UspPlan
    D = 128
    q, k, v = _usp_inputs(B, S, H, D, 450)
    plan = UspPlan(B, S, H, D, U, R, fp8_qv=True)
    out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), out)
    torch.cuda.synchronize()
    ref, _ = oatt.attention(_decoded(q), f64(k), _decoded(v))
    assert_bf16_close(f64(out), ref, "e4m3 Q/V")


def test_usp_e4m3_double_stream_with_rope():
    from sequence_attention_gb300.usp import UspPlan
    B, S, H, D, U, R, S_txt = 1, 700, 5, 128, 2, 2, 77
    qkv = _usp_inputs(B, S, H, D, 460)
    cos, sin = synth.rope_tables_joint(S_txt, S, D)
    plan = UspPlan(B, S, H, D, U, R, rope=(cos.cuda(), sin.cuda()), fp8_qv=True)
    txt = [t[:, :S_txt].contiguous().cuda() for t in qkv]
    img = [t[:, S_txt:].contiguous().cuda() for t in qkv]
    out_t = torch.empty((B, S_txt, H, D), dtype=torch.bfloat16, device="cuda")
    out_i = torch.empty((B, S - S_txt, H, D), dtype=torch.bfloat16, device="cuda")
    plan.run_joint(txt, img, out_t, out_i)
    torch.cuda.synchronize()
    c, s = cos.double().numpy(), sin.double().numpy()
    ref, _ = oatt.attention(orope.rope(_decoded(qkv[0]), c, s), orope.rope(f64(qkv[1]), c, s), _decoded(qkv[2]))
    got = np.concatenate([f64(out_t), f64(out_i)], axis=1)
    assert_bf16_close(got, ref, "e4m3 double-stream block")


def test_usp_e4m3_qvo_within_the_format_bound():
    # With O on the e4m3 wire too, each output element carries one more e4m3
    # rounding of at most 2^-4 of its magnitude (plus 2^-10 of its head's
    # scale below the normal range).  By the triangle inequality the
    # relative RMS against the oracle's attention over the decoded Q, V is
    # at most the bf16 bar plus 2^-4.
    from sequence_attention_gb300.usp import UspPlan
    B, S, H, D, U, R = 1, 700, 5, 128, 2, 2
    q, k, v = _usp_inputs(B, S, H, D, 470)
    plan = UspPlan(B, S, H, D, U, R, fp8_qv=True, fp8_o=True)
    out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), out)
    torch.cuda.synchronize()
    ref, _ = oatt.attention(_decoded(q), f64(k), _decoded(v))
    got = f64(out)
    assert np.all(np.isfinite(got))
    rr = rel_rms(got, ref)
    assert rr <= 5e-3 + 2.0 ** -4, rr
    amax = np.max(np.abs(ref), axis=-1, keepdims=True)
    assert np.all(np.abs(got - ref) <= 2e-2 + 2.0 ** -4 * amax * (1 + 2.0 ** -3))
