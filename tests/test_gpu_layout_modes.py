"""GPU parity of the alternate layouts: padding-free uneven heads (cache-dit
"Context Parallelism", Any Head Num without padding) and lcm(SP, 64)
sequence padding (xLLM "DiT Architecture and Capability Matrix").

The permutation buffers are compared bit for bit with the oracle; the
padding rows must be zero on the wire and in the head layout, must not be
rotated, and must never reach the output; attention end to end meets the
bf16 bars against the oracle's attention over the real rows.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import fp8 as ofp8
from oracle import layout as olayout
from oracle import rope as orope
from oracle import ulysses as ou
from tests.helpers import assert_bf16_close, assert_rotation_close, bits, f64

pytestmark = pytest.mark.gpu

MODES = [(False, False), (True, True), (False, True)]     # (pad_heads, pad_lcm64)
CASES = [
    # B, S, H, D, U, R
    (1, 17, 5, 8, 3, 1),
    (2, 37, 5, 16, 3, 2),
    (1, 20, 6, 16, 4, 2),      # lcm padding leaves the second ring block all padding
    (2, 24, 24, 16, 5, 2),
    (1, 1000, 6, 128, 4, 2),
    (1, 300, 30, 64, 4, 1),    # 30 heads over 4 ranks: 8, 8, 7, 7 without padding
]


def _layouts(case, mode):
    import sequence_attention_gb300 as sa
    return (sa.dit_sp_layout_init(*case, pad_heads=mode[0], pad_lcm64=mode[1]),
            olayout.make_layout(*case, pad_heads=mode[0], pad_lcm64=mode[1]))


def _rank_view(t, ref, r, v):
    return t[r, :, : ref.ring_len[r], ref.head_off[v]:ref.head_off[v] + ref.head_len[v]]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("mode", MODES)
def test_s2h_bit_exact(case, mode):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L, ref = _layouts(case, mode)
    planes = [synth.normal((B, S, H, D), 500 + p, 1.0, "bf16").cuda() for p in range(3)]
    send = torch.empty(L.wire_elems(3), dtype=torch.bfloat16, device="cuda")
    recv = torch.empty_like(send)
    heads = [torch.full(L.head_shape(), float("nan"), dtype=t, device="cuda")
             for t in (torch.bfloat16, torch.bfloat16, torch.float16)]
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 3, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, heads)
    torch.cuda.synchronize()
    o_send = ou.s2h_pack(ref, [bits(p) for p in planes], "bf16", "bf16")
    np.testing.assert_array_equal(bits(send), o_send)
    o_recv = ou.a2a(ref, "s2h", 3, o_send)
    np.testing.assert_array_equal(bits(recv), o_recv)
    for (r, v), pl in ou.s2h_unpack(ref, o_recv, "bf16", ("bf16", "bf16", "f16")).items():
        for p in range(3):
            np.testing.assert_array_equal(bits(_rank_view(heads[p], ref, r, v)), pl[p])


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("mode", MODES)
def test_h2s_bit_exact_with_garbage_in_the_padding(case, mode):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L, ref = _layouts(case, mode)
    head = synth.normal(L.head_shape(), 510, 1.0, "bf16").cuda()
    for r in range(R):                         # NaN in every padding row
        head[r, :, ref.real_rows(r):] = float("nan")
    send = torch.empty(L.wire_elems(1), dtype=torch.bfloat16, device="cuda")
    recv = torch.empty_like(send)
    out = torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [head], send)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_HEAD_TO_SEQ, recv, [out])
    torch.cuda.synchronize()
    hb = bits(head)
    o_ranks = {(r, v): _rank_view(hb, ref, r, v) for r in range(R) for v in range(U)}
    o_send = ou.h2s_pack(ref, o_ranks, "bf16", "bf16")
    np.testing.assert_array_equal(bits(send), o_send)
    np.testing.assert_array_equal(bits(out), ou.h2s_unpack(ref, ou.a2a(ref, "h2s", 1, o_send), "bf16", "bf16"))
    assert not torch.isnan(out).any()


@pytest.mark.parametrize("case", [c for c in CASES if c[3] >= 16])
@pytest.mark.parametrize("mode", MODES)
def test_e4m3_wire_bit_exact(case, mode):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L, ref = _layouts(case, mode)
    planes = [synth.normal((B, S, H, D), 520 + p, 1.0, "bf16").cuda() for p in range(2)]
    send = torch.empty(L.wire_bytes_e4m3(2), dtype=torch.uint8, device="cuda")
    recv = torch.empty_like(send)
    heads = [torch.full(L.head_shape(), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 2, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, heads)
    torch.cuda.synchronize()
    o_send = ofp8.s2h_pack(ref, [bits(p) for p in planes], "bf16")
    np.testing.assert_array_equal(send.cpu().numpy(), o_send.view(np.uint8))
    o_recv = ofp8.a2a(ref, "s2h", 2, o_send)
    for (r, v), pl in ofp8.s2h_unpack(ref, o_recv, ["bf16", "bf16"]).items():
        for p in range(2):
            np.testing.assert_array_equal(bits(_rank_view(heads[p], ref, r, v)), pl[p])


@pytest.mark.parametrize("case", [CASES[2], CASES[4]])
def test_rope_leaves_padding_rows_alone(case):
    # the angle tables hold the S real rows only
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L, ref = _layouts(case, (True, True))
    planes = [synth.normal((B, S, H, D), 530 + p, 1.0, "bf16").cuda() for p in range(2)]
    send = torch.empty(L.wire_elems(2), dtype=torch.bfloat16, device="cuda")
    recv = torch.empty_like(send)
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 2, send, recv)
    cos, sin = synth.rope_tables_linear(S, D)
    heads = [torch.full(L.head_shape(), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    sa.dit_ulysses_unpack_rope(L, recv, heads, cos.cuda(), sin.cuda(), 0b11)
    torch.cuda.synchronize()
    cpad = np.concatenate([cos.double().numpy(), np.ones((ref.S_pad - S, D // 2))])
    spad = np.concatenate([sin.double().numpy(), np.zeros((ref.S_pad - S, D // 2))])
    want = orope.receive_prep(ref, bits(recv), "bf16", ["bf16", "bf16"], cpad, spad, 0b11)
    xin = ou.s2h_unpack(ref, bits(recv), "bf16", ["bf16", "bf16"])
    from oracle import numeric
    for (r, v), pl in want.items():
        for p in range(2):
            x = numeric.to_f64(xin[(r, v)][p], "bf16")
            got = f64(_rank_view(heads[p], ref, r, v))
            assert_rotation_close(got, pl[p], x, "bf16", f"rank ({r},{v})")
            assert np.all(got[:, ref.real_rows(r):] == 0)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("B,S,H,U,R", [(1, 700, 5, 2, 2), (1, 20, 6, 4, 2), (2, 517, 30, 4, 1), (1, 333, 7, 3, 2)])
def test_usp_in_every_layout(mode, B, S, H, U, R):
    from sequence_attention_gb300.usp import UspPlan
    D = 128
    q, k, v = (synth.normal((B, S, H, D), 540 + p, 0.5, "bf16") for p in range(3))
    plan = UspPlan(B, S, H, D, U, R, pad_heads=mode[0], pad_lcm64=mode[1])
    out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), out)
    torch.cuda.synchronize()
    ref, _ = oatt.attention(f64(q), f64(k), f64(v))
    assert_bf16_close(f64(out), ref, f"USP {mode}")


@pytest.mark.parametrize("name,U,mode", [("qwen1328", 5, (False, False)), ("wan", 8, (True, True)),
                                         ("flux1008", 4, (False, True)), ("qwen1328", 5, (False, True))])
def test_full_size_layout_modes(name, U, mode):
    """At the workloads' full sizes in the alternate layouts: S2H gives every
    rank exactly its rows and heads of the global tensors (padding rows and
    padded heads zero), and H2S after S2H is the identity, bit for bit."""
    import sequence_attention_gb300 as sa
    w = synth.WORKLOADS[name]
    L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, U, w.R, pad_heads=mode[0], pad_lcm64=mode[1])
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
            m = L.real_rows(r)
            got = heads[p][r, :, :m, : w.H]
            assert torch.equal(got.view(torch.int16), x[:, L.ring_off[r]:L.ring_off[r] + m].view(torch.int16))
            assert not heads[p][r, :, m:L.ring_len[r]].any()            # padding rows are zero
        assert not heads[p][..., w.H:, :].any()                          # padded heads are zero
    out = torch.empty_like(q)
    s1 = torch.empty(L.wire_elems(1), dtype=torch.bfloat16, device="cuda")
    r1 = torch.empty_like(s1)
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [heads[1]], s1)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, s1, r1)
    sa.dit_ulysses_unpack(L, sa.DIT_HEAD_TO_SEQ, r1, [out])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), k.view(torch.int16))
