"""GPU parity of the one-pass seq<->head permutation (dit_ulysses_seq_to_head,
dit_ulysses_head_to_seq) against the oracle, bit for bit.

On one memory the exchange aliases receive and send blocks, so the one-pass
result must equal the oracle's explicit pack -> alltoallv -> unpack index
permutation with the wire in the source type (edge-dit.cpp "Parallel
execution", packed QKV send path and head-to-sequence path; SGLang Diffusion
"Parallelism Overview", The Ulysses transport).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import layout as olayout
from oracle import rope as orope
from oracle import ulysses as ou
from tests.helpers import DT_NAME, assert_rotation_close, bits

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
    (3, 129, 7, 16, 4, 3),     # B = 3, three ring blocks, ragged everything
]
FLAGS = [(True, False), (False, False), (True, True), (False, True)]   # (pad_heads, pad_lcm64)


def _oracle_heads(ref, planes_bits, in_dt, dst_dts):
    """Oracle head layout {(r, v): [planes]} of pack -> a2a -> unpack with
    the wire in the source type."""
    send = ou.s2h_pack(ref, planes_bits, in_dt, in_dt)
    recv = ou.a2a(ref, "s2h", len(planes_bits), send)
    return ou.s2h_unpack(ref, recv, in_dt, dst_dts)


def _check_heads(L, ref, heads, o_ranks):
    hb = [bits(h) for h in heads]
    for (r, v), pl in o_ranks.items():
        h0, n = ref.head_off[v], ref.head_len[v]
        for p in range(len(heads)):
            got = hb[p][r, :, : ref.ring_len[r], h0:h0 + n]
            np.testing.assert_array_equal(got, pl[p], err_msg=f"plane {p}, ring block {r}, group {v}")


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("dts", [("bf16", ("bf16", "bf16", "f16")), ("f32", ("f32", "f32", "f32")),
                                 ("f32", ("bf16", "bf16", "bf16")), ("bf16", ("f32", "f32", "f32"))])
def test_seq_to_head_bit_exact(case, flags, dts):
    import sequence_attention_gb300 as sa
    in_dt, dst_dts = dts
    B, S, H, D, U, R = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R, *flags)
    ref = olayout.make_layout(B, S, H, D, U, R, *flags)
    planes = [synth.normal((B, S, H, D), 300 + p, 1.0, in_dt) for p in range(3)]
    heads = [torch.full(L.head_shape(), float("nan"), dtype=synth.torch_dtype(dt), device="cuda")
             for dt in dst_dts]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_seq_to_head(L, [p.cuda() for p in planes], heads, flag)
    torch.cuda.synchronize()
    _check_heads(L, ref, heads, _oracle_heads(ref, [bits(p) for p in planes], in_dt, dst_dts))
    # rows past each ring block's length are never written
    for r in range(R):
        assert torch.isnan(heads[0][r, :, ref.ring_len[r]:].float()).all()
    assert int(flag.item()) == 0


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("dts", [("bf16", "bf16"), ("f32", "bf16"), ("f16", "f32")])
def test_head_to_seq_bit_exact(case, flags, dts):
    """NaN in the head layout's padded heads and padding rows never reaches
    the output; every real element equals the oracle's."""
    import sequence_attention_gb300 as sa
    src_dt, out_dt = dts
    B, S, H, D, U, R = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R, *flags)
    ref = olayout.make_layout(B, S, H, D, U, R, *flags)
    head = synth.normal(L.head_shape(), 9, 1.0, src_dt)
    head[..., H:, :] = float("nan")                       # padded heads
    for r in range(R):
        head[r, :, ref.real_rows(r):] = float("nan")        # padding rows and the rest
    out = torch.full((B, S, H, D), 7.0, dtype=synth.torch_dtype(out_dt), device="cuda")
    sa.dit_ulysses_head_to_seq(L, head.cuda(), out)
    torch.cuda.synchronize()
    hb = bits(head)
    o_ranks = {(r, v): hb[r, :, : ref.ring_len[r], ref.head_off[v]:ref.head_off[v] + ref.head_len[v]]
               for r in range(R) for v in range(U)}
    o_recv = ou.a2a(ref, "h2s", 1, ou.h2s_pack(ref, o_ranks, src_dt, src_dt))
    np.testing.assert_array_equal(bits(out), ou.h2s_unpack(ref, o_recv, src_dt, out_dt))
    assert not torch.isnan(out.float()).any()


@pytest.mark.parametrize("case", CASES[:7])
def test_round_trip_is_identity(case):
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    for flags in FLAGS:
        L = sa.dit_sp_layout_init(B, S, H, D, U, R, *flags)
        x = synth.normal((B, S, H, D), 5, 1.0, "bf16").cuda()
        head = torch.full(L.head_shape(), float("nan"), dtype=torch.bfloat16, device="cuda")
        out = torch.empty_like(x)
        sa.dit_ulysses_seq_to_head(L, [x], [head])
        sa.dit_ulysses_head_to_seq(L, head, out)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), x.view(torch.int16))


@pytest.mark.parametrize("case,flags", [((1, 700, 5, 128, 2, 2), (True, False)), ((2, 517, 4, 64, 3, 1), (False, True)),
                                        ((1, 37, 5, 8, 3, 2), (True, True))])
@pytest.mark.parametrize("S_txt", [0, 1, 77, "S"])
def test_paired_streams_equal_the_joint_tensor(case, flags, S_txt):
    """Text rows from one tensor and image rows from another give the same
    head layout as the concatenated joint sequence, and the head-to-seq pass
    writes each output row back to its stream (FLUX double-stream blocks)."""
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    S_txt = S if S_txt == "S" else min(S_txt, S)
    L = sa.dit_sp_layout_init(B, S, H, D, U, R, *flags)
    joint = [synth.normal((B, S, H, D), 40 + p, 1.0, "bf16").cuda() for p in range(3)]
    ref = [torch.empty(L.head_shape(), dtype=t, device="cuda") for t in (torch.bfloat16, torch.bfloat16, torch.float16)]
    got = [torch.empty_like(t) for t in ref]
    sa.dit_ulysses_seq_to_head(L, joint, ref)
    txt = [j[:, :S_txt].contiguous() for j in joint]
    img = [j[:, S_txt:].contiguous() for j in joint]
    first, second = (txt, img) if 0 < S_txt < S else ((img, None) if S_txt == 0 else (txt, None))
    sa.dit_ulysses_seq_to_head(L, first, got, src2=second)
    out_t = torch.full((B, S_txt, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    out_i = torch.full((B, S - S_txt, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    if 0 < S_txt < S:
        sa.dit_ulysses_head_to_seq(L, ref[0], out_t, out_i)
    elif S_txt == 0:
        sa.dit_ulysses_head_to_seq(L, ref[0], out_i)
    else:
        sa.dit_ulysses_head_to_seq(L, ref[0], out_t)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        for r in range(R):
            n = L.ring_len[r]
            assert torch.equal(a[r, :, :n].view(torch.int16), b[r, :, :n].view(torch.int16))
    back = torch.cat([out_t, out_i], dim=1)
    assert torch.equal(back.view(torch.int16), joint[0].view(torch.int16))


@pytest.mark.parametrize("case", [(1, 700, 5, 128, 2, 2), (2, 129, 3, 64, 4, 1), (1, 333, 6, 32, 3, 3)])
@pytest.mark.parametrize("flags", [(True, False), (False, True)])
def test_rope_matches_the_receive_preparation(case, flags):
    """With RoPE on Q and K, the one-pass layout equals the three-call path
    that ends in dit_ulysses_unpack_rope bit for bit (the same fp32
    arithmetic), and the oracle's fp64 rotation within the rotation bound."""
    import sequence_attention_gb300 as sa
    B, S, H, D, U, R = case
    L = sa.dit_sp_layout_init(B, S, H, D, U, R, *flags)
    ref = olayout.make_layout(B, S, H, D, U, R, *flags)
    planes = [synth.normal((B, S, H, D), 60 + p, 1.0, "bf16") for p in range(3)]
    cos, sin = synth.rope_tables_linear(S, D)
    dts = (torch.bfloat16, torch.bfloat16, torch.float16)
    direct = [torch.empty(L.head_shape(), dtype=t, device="cuda") for t in dts]
    three = [torch.empty_like(t) for t in direct]
    dp = [p.cuda() for p in planes]
    sa.dit_ulysses_seq_to_head(L, dp, direct, rope=(cos.cuda(), sin.cuda()), rope_planes=0b011)
    send = torch.empty(L.wire_elems(3), dtype=torch.bfloat16, device="cuda")
    recv = torch.empty_like(send)
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, dp, send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 3, send, recv)
    sa.dit_ulysses_unpack_rope(L, recv, three, cos.cuda(), sin.cuda(), 0b011)
    torch.cuda.synchronize()
    for a, b in zip(direct, three):
        for r in range(R):
            n = L.ring_len[r]
            assert torch.equal(a[r, :, :n].view(torch.int16), b[r, :, :n].view(torch.int16))
            # padded heads are not rotated: +0 bits in both paths
            assert not a[r, :, :n, H:].view(torch.int16).any()
    o_send = ou.s2h_pack(ref, [bits(p) for p in planes], "bf16", "bf16")
    o_recv = ou.a2a(ref, "s2h", 3, o_send)
    o_ranks = orope.receive_prep(ref, o_recv, "bf16", ["bf16", "bf16", "f16"], cos.double().numpy(),
                                 sin.double().numpy(), 0b011)
    unrot = ou.s2h_unpack(ref, o_recv, "bf16", ["bf16", "bf16", "bf16"])
    for (r, v), pl in o_ranks.items():
        h0, n = ref.head_off[v], ref.head_len[v]
        for p in (0, 1):
            got = direct[p][r, :, : ref.ring_len[r], h0:h0 + n].float().cpu().double().numpy()
            x = unrot[(r, v)][p].view(np.uint16).astype(np.uint32) << 16
            assert_rotation_close(got, pl[p], x.view(np.float32), "bf16", f"plane {p}")
        np.testing.assert_array_equal(bits(direct[2][r, :, : ref.ring_len[r], h0:h0 + n]), pl[2])


def test_range_flag_on_f16_overflow():
    import sequence_attention_gb300 as sa
    L = sa.dit_sp_layout_init(1, 16, 4, 8, 2, 1)
    planes = [synth.normal((1, 16, 4, 8), 1 + p, 1.0, "bf16").cuda() for p in range(3)]
    dts = (torch.bfloat16, torch.bfloat16, torch.float16)
    heads = [torch.empty(L.head_shape(), dtype=t, device="cuda") for t in dts]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_seq_to_head(L, planes, heads, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    planes[2][0, 3, 1, 2] = 1.0e6          # representable in bf16, not in f16
    sa.dit_ulysses_seq_to_head(L, planes, heads, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 5            # DIT_ERR_RANGE
    assert torch.isinf(heads[2][0, 0, 3, 1, 2].float())


@pytest.mark.parametrize("name,U", [("flux1024", 2), ("flux1024", 4), ("flux1008", 4), ("flux1008_4480", 4),
                                    ("qwen1328", 5)])
def test_full_size_against_the_oracle(name, U):
    """At the workloads' full sizes, in the launch configuration the bench
    times: the one-pass head layout equals the oracle's pack -> alltoallv ->
    unpack bit for bit in every plane (V to f16), and the one-pass head-to-seq
    of an output-like head tensor equals the oracle's inverse."""
    import sequence_attention_gb300 as sa
    w = synth.WORKLOADS[name]
    L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, U, w.R)
    ref = olayout.make_layout(w.B, w.S, w.H, w.D, U, w.R)
    planes = w.qkv()
    dts = ("bf16", "bf16", "f16")
    heads = [torch.empty(L.head_shape(), dtype=synth.torch_dtype(dt), device="cuda") for dt in dts]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_seq_to_head(L, [p.cuda() for p in planes], heads, flag)
    torch.cuda.synchronize()
    _check_heads(L, ref, heads, _oracle_heads(ref, [bits(p) for p in planes], "bf16", dts))
    assert int(flag.item()) == 0
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    sa.dit_ulysses_head_to_seq(L, heads[0], out)
    torch.cuda.synchronize()
    hb = bits(heads[0])
    o_ranks = {(r, v): hb[r, :, : ref.ring_len[r], ref.head_off[v]:ref.head_off[v] + ref.head_len[v]]
               for r in range(ref.R) for v in range(U)}
    o_recv = ou.a2a(ref, "h2s", 1, ou.h2s_pack(ref, o_ranks, "bf16", "bf16"))
    np.testing.assert_array_equal(bits(out), ou.h2s_unpack(ref, o_recv, "bf16", "bf16"))
    np.testing.assert_array_equal(bits(out), bits(planes[0]))


def test_full_size_wan():
    """Wan-like (B1 S75600 H40 D128, U=8, R=4): rank (r, v) holds exactly its
    slice of the global tensors, padded heads are zero, and the head-to-seq
    pass restores the input bit for bit (checked on the device)."""
    import sequence_attention_gb300 as sa
    w = synth.WORKLOADS["wan"]
    L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, 8, w.R)
    q, k, v = w.qkv("cuda")
    heads = [torch.empty(L.head_shape(), dtype=t, device="cuda") for t in (torch.bfloat16, torch.bfloat16, torch.float16)]
    sa.dit_ulysses_seq_to_head(L, [q, k, v], heads)
    for p, x in enumerate((q, k, v)):
        for r in range(L.R):
            rows = slice(L.ring_off[r], L.ring_off[r] + L.ring_len[r])
            got = heads[p][r, :, : L.ring_len[r], : w.H]
            want = x[:, rows] if p < 2 else x[:, rows].to(torch.float16)
            assert torch.equal(got.view(torch.int16), want.contiguous().view(torch.int16))
        assert not heads[p][..., w.H:, :].any()
    out = torch.empty_like(q)
    sa.dit_ulysses_head_to_seq(L, heads[0], out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), q.view(torch.int16))
