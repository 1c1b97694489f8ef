"""Full-size parity in the launch configurations the benchmark times.

* Every row and head of the FLUX-1024-like (U = 2 and 4) and FLUX-1008-like
  (S = 4481 and 4480, U = 4, R = 2) steps against the fp64 oracle's
  attention over the whole sequence (edge-dit.cpp "Parallel execution",
  Ulysses sequence parallelism: the split attention is exact; SGLang
  Diffusion "Parallelism Overview", What happens to the shapes), through
  both the one-pass layout and the pack / exchange / unpack calls.
* The receive preparation with RoPE (edge-dit.cpp, receive preparation) on
  the FLUX-like joint sequence (4096 image + 512 text tokens, U = 4) and on
  the first ring block of the Wan-like shape (U = 8, R = 4).
* The e4m3 wire of Q and V (cache-dit "Context Parallelism", Async FP8
  Ulysses Attention) at the same two sizes, bit for bit.

A Wan-size launch is checked on its first ring block: the ranks of ring
block 0 come first in every wire order and in the head layout, and their
buffers equal those of the layout of ring block 0 alone (S = 18900, R = 1),
which the oracle computes in seconds.
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
from oracle import ulysses as ou
from tests.helpers import assert_bf16_close, assert_rotation_close, bits, f64

pytestmark = pytest.mark.gpu

_ORACLE = {}


def _oracle_attention(name):
    """fp64 attention of the whole workload, one head at a time (cached)."""
    if name not in _ORACLE:
        w = synth.WORKLOADS[name]
        q, k, v = w.qkv()
        out = np.empty((w.B, w.S, w.H, w.D))
        for b in range(w.B):
            for h in range(w.H):
                o, _ = oatt.attention(f64(q[b:b + 1, :, h:h + 1]), f64(k[b:b + 1, :, h:h + 1]),
                                      f64(v[b:b + 1, :, h:h + 1]))
                out[b, :, h] = o[0, :, 0]
        _ORACLE[name] = out
    return _ORACLE[name]


@pytest.mark.parametrize("exchange,ring_merge", [("direct", "fold"), ("a2a", "partials")])
@pytest.mark.parametrize("name,U", [("flux1024", 2), ("flux1024", 4), ("flux1008", 4), ("flux1008_4480", 4)])
def test_every_row_against_the_full_oracle(name, U, exchange, ring_merge):
    from sequence_attention_gb300.usp import UspPlan
    w = synth.WORKLOADS[name]
    q, k, v = w.qkv()
    plan = UspPlan(w.B, w.S, w.H, w.D, U, w.R, exchange=exchange, ring_merge=ring_merge)
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), out, check=True)
    assert_bf16_close(f64(out), _oracle_attention(name), f"{name} U={U} {exchange}")


def _wan_block0():
    w = synth.WORKLOADS["wan"]
    return w, (w.B, w.S, w.H, w.D, 8, w.R), (w.B, w.S // w.R, w.H, w.D, 8, 1)


def _joint_tables(S_txt, S, D):
    cos, sin = synth.rope_tables_joint(S_txt, S, D)
    return cos, sin


@pytest.mark.parametrize("path", ["unpack_rope", "seq_to_head"])
@pytest.mark.parametrize("size", ["flux", "wan_block0"])
def test_receive_prep_rope_at_workload_size(path, size):
    """Rotated Q and K within the fp32-then-round bound of the oracle's fp64
    rotation, V (f16) bit for bit, at the sizes the bench times."""
    import sequence_attention_gb300 as sa
    if size == "flux":
        w = synth.WORKLOADS["flux1024"]
        big = small = (w.B, w.S, w.H, w.D, 4, 1)
        S_txt = w.S_txt
    else:
        w, big, small = _wan_block0()
        S_txt = 0
    L = sa.dit_sp_layout_init(*big)
    ref = olayout.make_layout(*small)
    q, k, v = w.qkv()
    cos, sin = _joint_tables(S_txt, w.S, w.D)
    heads = [torch.empty(L.head_shape(), dtype=t, device="cuda") for t in (torch.bfloat16, torch.bfloat16, torch.float16)]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    if path == "unpack_rope":
        send = torch.empty(L.wire_elems(3), dtype=torch.bfloat16, device="cuda")
        recv = torch.empty_like(send)
        sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, [q.cuda(), k.cuda(), v.cuda()], send)
        sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 3, send, recv)
        del send
        sa.dit_ulysses_unpack_rope(L, recv, heads, cos.cuda(), sin.cuda(), 0b011, flag)
        del recv
    else:
        sa.dit_ulysses_seq_to_head(L, [q.cuda(), k.cuda(), v.cuda()], heads, flag, rope=(cos.cuda(), sin.cuda()))
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    Sr = ref.S
    planes = [bits(t[:, :Sr]) for t in (q, k, v)]
    o_recv = ou.a2a(ref, "s2h", 3, ou.s2h_pack(ref, planes, "bf16", "bf16"))
    c, s = cos[:Sr].double().numpy(), sin[:Sr].double().numpy()
    want = orope.receive_prep(ref, o_recv, "bf16", ["bf16", "bf16", "f16"], c, s, 0b011)
    xin = ou.s2h_unpack(ref, o_recv, "bf16", ["bf16", "bf16", "bf16"])
    for (r, vv), pl in want.items():
        sl = (r, slice(None), slice(0, ref.ring_len[r]), slice(vv * ref.Hl, (vv + 1) * ref.Hl))
        for p in range(2):
            x = numeric.to_f64(xin[(r, vv)][p], "bf16")
            assert_rotation_close(f64(heads[p][sl]), pl[p], x, "bf16", f"plane {p} rank ({r},{vv})")
        np.testing.assert_array_equal(bits(heads[2][sl]), pl[2])


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


@pytest.mark.parametrize("size", ["flux", "wan_block0"])
def test_e4m3_wire_at_workload_size(size):
    """Quantizing pack of Q and V, the exchange of the records and the
    decoding unpack (V to f16), each bit for bit against the oracle, in the
    launch configuration of the bench (FLUX-like U = 4; Wan-like U = 8,
    R = 4, first ring block)."""
    import sequence_attention_gb300 as sa
    if size == "flux":
        w = synth.WORKLOADS["flux1024"]
        big = small = (w.B, w.S, w.H, w.D, 4, 1)
    else:
        w, big, small = _wan_block0()
    L = sa.dit_sp_layout_init(*big)
    ref = olayout.make_layout(*small)
    q, _, v = w.qkv()
    send = torch.empty(L.wire_bytes_e4m3(2), dtype=torch.uint8, device="cuda")
    recv = torch.empty_like(send)
    heads = [torch.empty(L.head_shape(), dtype=torch.bfloat16, device="cuda"),
             torch.empty(L.head_shape(), dtype=torch.float16, device="cuda")]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, [q.cuda(), v.cuda()], send)
    sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 2, send, recv)
    sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, heads, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    Sr = ref.S
    o_send = ofp8.s2h_pack(ref, [bits(q[:, :Sr]), bits(v[:, :Sr])], "bf16").view(np.uint8)
    n = o_send.size                              # ring block 0's records come first
    np.testing.assert_array_equal(_bytes(send[:n]), o_send)
    o_recv = ofp8.a2a(ref, "s2h", 2, o_send.view(np.uint16))
    np.testing.assert_array_equal(_bytes(recv[:n]), o_recv.view(np.uint8))
    for (r, vv), pl in ofp8.s2h_unpack(ref, o_recv, ["bf16", "f16"]).items():
        for p in range(2):
            got = bits(heads[p][r, :, : ref.ring_len[r], vv * ref.Hl:(vv + 1) * ref.Hl])
            np.testing.assert_array_equal(got, pl[p])
    # the output direction at the same size: O on the e4m3 wire, back to bf16
    head = torch.empty(L.head_shape(), dtype=torch.bfloat16, device="cuda")
    head.copy_(heads[0])
    send_o = torch.empty(L.wire_bytes_e4m3(1), dtype=torch.uint8, device="cuda")
    recv_o = torch.empty_like(send_o)
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_HEAD_TO_SEQ, [head], send_o)
    sa.dit_a2a_sim(L, sa.DIT_HEAD_TO_SEQ, 1, send_o, recv_o)
    sa.dit_ulysses_unpack(L, sa.DIT_HEAD_TO_SEQ, recv_o, [out])
    torch.cuda.synchronize()
    hb = bits(head[:1]) if size != "flux" else bits(head)
    o_ranks = {(r, vv): hb[r, :, : ref.ring_len[r], vv * ref.Hl:(vv + 1) * ref.Hl]
               for r in range(ref.R) for vv in range(ref.U)}
    o_send1 = ofp8.h2s_pack(ref, o_ranks, "bf16")
    n1 = o_send1.view(np.uint8).size
    np.testing.assert_array_equal(_bytes(send_o[:n1]), o_send1.view(np.uint8))
    o_recv1 = ofp8.a2a(ref, "h2s", 1, o_send1)
    np.testing.assert_array_equal(_bytes(recv_o[:n1]), o_recv1.view(np.uint8))
    np.testing.assert_array_equal(bits(out[:, :Sr]), ofp8.h2s_unpack(ref, o_recv1, "bf16"))
