"""GPU parity of packed variable-length attention and of the masked
(tail-padded) text path against the oracle.

Varlen: every sequence of the packed rows attends only to its own keys
(the oracle's block-diagonal definition), through dit_attn_varlen, on both
the tensor-core and the fp32 path.  Masked text: the joint sequence
[text with tail padding; image] is attended as two key blocks of one
dit_attn_partial call (the padding trimmed by the text block's length) and
folded with dit_attn_merge_lse, as the pages fold the text portion into the
rest, against the oracle's masked attention.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from tests.helpers import F32_MAX_ABS, LSE_ABS, assert_bf16_close, f64, max_abs

pytestmark = pytest.mark.gpu

SEGMENTS = [
    # (cu_q, cu_k)
    ([0, 300], [0, 300]),
    ([0, 129, 129, 700, 701], [0, 64, 320, 320, 1000]),        # empty query and empty key segments
    ([0, 1000, 1256, 3000], [0, 1000, 1256, 3000]),
    ([5, 133, 260], [3, 70, 390]),                               # offsets that start past row 0
    (list(range(0, 1300, 100)), list(range(0, 1300, 100))),      # 12 segments: two launches
]


def _packed(T, H, D, seed, dt, scale=0.5):
    return synth.normal((T, H, D), seed, scale, dt)


@pytest.mark.parametrize("segs", SEGMENTS)
@pytest.mark.parametrize("D,vdt,odt", [(128, "f16", "bf16"), (64, "bf16", "f32"), (128, "f16", "f32")])
def test_varlen_tensor_cores(segs, D, vdt, odt):
    import sequence_attention_gb300 as sa
    cu_q, cu_k = segs
    H = 3
    Tq, Tk = cu_q[-1] + 7, cu_k[-1] + 5                         # rows past the last sequence
    q = _packed(Tq, H, D, 600, "bf16")
    k = _packed(Tk, H, D, 601, "bf16")
    v = _packed(Tk, H, D, 602, vdt)
    o = torch.full((Tq, H, D), float("nan"), dtype=synth.torch_dtype(odt), device="cuda")
    lse = torch.full((H, Tq), float("nan"), dtype=torch.float32, device="cuda")
    sa.dit_attn_varlen(q.cuda(), k.cuda(), v.cuda(), o, cu_q, cu_k, lse)
    torch.cuda.synchronize()
    ref, lref = oatt.varlen(f64(q), f64(k), f64(v), cu_q, cu_k)
    got, lg = f64(o), lse.cpu().double().numpy()
    for s in range(len(cu_q) - 1):
        rows = slice(cu_q[s], cu_q[s + 1])
        if cu_q[s + 1] == cu_q[s]:
            continue
        if cu_k[s + 1] == cu_k[s]:
            assert np.all(got[rows] == 0) and np.all(np.isneginf(lg[:, rows]))
            continue
        assert_bf16_close(got[rows], ref[rows], f"segment {s}")
        assert np.max(np.abs(lg[:, rows] - lref[:, rows])) <= 2e-3
    # rows outside every sequence are untouched
    outside = np.ones(Tq, bool)
    for s in range(len(cu_q) - 1):
        outside[cu_q[s]:cu_q[s + 1]] = False
    assert np.all(np.isnan(got[outside]))


@pytest.mark.parametrize("segs", SEGMENTS[1:4])
def test_varlen_fp32(segs):
    import sequence_attention_gb300 as sa
    cu_q, cu_k = segs
    H, D = 2, 64
    q = _packed(cu_q[-1], H, D, 610, "f32", 1.0)
    k = _packed(cu_k[-1], H, D, 611, "f32", 1.0)
    v = _packed(cu_k[-1], H, D, 612, "f32", 1.0)
    o = torch.zeros((cu_q[-1], H, D), dtype=torch.float32, device="cuda")
    lse = torch.zeros((H, cu_q[-1]), dtype=torch.float32, device="cuda")
    sa.dit_attn_varlen(q.cuda(), k.cuda(), v.cuda(), o, cu_q, cu_k, lse)
    torch.cuda.synchronize()
    ref, lref = oatt.varlen(f64(q), f64(k), f64(v), cu_q, cu_k)
    live = np.zeros(cu_q[-1], bool)
    for s in range(len(cu_q) - 1):
        if cu_k[s + 1] > cu_k[s]:
            live[cu_q[s]:cu_q[s + 1]] = True
    assert max_abs(f64(o)[live], ref[live]) <= F32_MAX_ABS
    assert np.max(np.abs(lse.cpu().double().numpy()[:, live] - lref[:, live])) <= LSE_ABS


def test_varlen_rejects_decreasing_offsets():
    import sequence_attention_gb300 as sa
    x = torch.zeros((10, 1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa.DitError):
        sa.dit_attn_varlen(x, x, x, x.clone(), [0, 5, 4], [0, 5, 10])


@pytest.mark.parametrize("B,S_txt,S_img,H,txt_len", [(2, 512, 1024, 4, [77, 300]), (1, 256, 700, 3, [256])])
def test_masked_text_by_two_key_blocks_and_merge(B, S_txt, S_img, H, txt_len):
    import sequence_attention_gb300 as sa
    D = 128
    S = S_txt + S_img
    q, k, v = (synth.normal((B, S, H, D), 620 + i, 0.5, "bf16") for i in range(3))
    qd, kd, vd = q.cuda(), k.cuda(), v.float().half().cuda()
    out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    for b in range(B):                      # the text length differs per prompt
        parts = torch.empty((1, 2, 1, S, H, D), dtype=torch.float32, device="cuda")
        lse = torch.empty((1, 2, 1, H, S), dtype=torch.float32, device="cuda")
        # key block 0 = the text rows (trimmed to the prompt's length), block 1 = the image rows
        kb = kd[b:b + 1].as_strided((2, 1, S_img, H, D), (S_txt * H * D, S * H * D, H * D, D, 1))
        vb = vd[b:b + 1].as_strided((2, 1, S_img, H, D), (S_txt * H * D, S * H * D, H * D, D, 1))
        sa.dit_attn_partial(qd[b:b + 1].unsqueeze(0), kb, vb, parts, lse, q_len=[S],
                            kv_len=[txt_len[b], S_img])
        sa.dit_attn_merge_lse(parts, lse, out[b:b + 1].unsqueeze(0))
    torch.cuda.synchronize()
    mask = np.ones((B, S), bool)
    for b in range(B):
        mask[b, txt_len[b]:S_txt] = False
    ref, _ = oatt.masked(f64(q), f64(k), f64(v.float().half()), mask)
    assert_bf16_close(f64(out), ref, "masked text")
