"""The whole hot path on the five workloads, against the fp64 oracle.

Each run goes seq-sharded Q/K/V -> Ulysses pack -> simulated all-to-all ->
unpack (V to f16) -> all ring partials in one launch -> log-sum-exp merge ->
inverse all-to-all -> seq-sharded output, through the C ABI.  Small cases are
compared in full; full-size cases on the first and last rows of every virtual
rank (the UAA and ring seams) plus seeded random rows, all heads, against the
oracle's attention over the full key sequence.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import layout as olayout
from oracle import usp as ousp
from tests.helpers import F32_MAX_ABS, assert_bf16_close, f64, max_abs, sample_rows

pytestmark = pytest.mark.gpu


def _plan(w, U, R=None, **kw):
    from sequence_attention_gb300.usp import UspPlan
    return UspPlan(w.B, w.S, w.H, w.D, U, w.R if R is None else R,
                   in_dtype=synth.torch_dtype(w.dtype), **kw)


def _oracle_rows(q, k, v, rows):
    """fp64 attention of the given query rows against all keys, head by head."""
    B, S, H, D = q.shape
    out = np.empty((B, len(rows), H, D))
    sel = torch.from_numpy(rows)
    for b in range(B):
        for h in range(H):
            qh = f64(q[b:b + 1, sel, h:h + 1])
            kh = f64(k[b:b + 1, :, h:h + 1])
            vh = f64(v[b:b + 1, :, h:h + 1])
            o, _ = oatt.attention(qh, kh, vh)
            out[b, :, h] = o[0, :, 0]
    return out


@pytest.mark.parametrize("U,R", [(2, 1), (1, 2), (2, 2)])
def test_tiny_fp32_full(U, R):
    w = synth.WORKLOADS["tiny"]
    q, k, v = w.qkv()
    plan = _plan(w, U, R)
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.float32, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), out)
    torch.cuda.synchronize()
    ref, _ = oatt.attention(f64(q), f64(k), f64(v))
    assert max_abs(f64(out), ref) <= F32_MAX_ABS
    # and the oracle's own USP composition agrees with its single shot
    o2, _ = ousp.usp_attention(olayout.make_layout(w.B, w.S, w.H, w.D, U, R), f64(q), f64(k), f64(v))
    assert max_abs(o2, ref) <= 1e-12


@pytest.mark.parametrize("exchange", ["direct", "a2a"])
@pytest.mark.parametrize("B,S,H,U,R", [(1, 1000, 5, 3, 2), (2, 700, 4, 2, 3), (1, 333, 3, 4, 1)])
def test_medium_bf16_full(B, S, H, U, R, exchange):
    """Sizes the oracle finishes in seconds, spanning several tiles and ragged
    tails, with padded heads and uneven ranks: compared in full."""
    D = 128
    q = synth.normal((B, S, H, D), 20, 0.5, "bf16")
    k = synth.normal((B, S, H, D), 21, 0.5, "bf16")
    v = synth.normal((B, S, H, D), 22, 0.5, "bf16")
    from sequence_attention_gb300.usp import UspPlan
    plan = UspPlan(B, S, H, D, U, R, exchange=exchange)
    out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), out, check=True)
    ref, _ = oatt.attention(f64(q), f64(k), f64(v))
    assert_bf16_close(f64(out), ref, "usp")


# FLUX-1024 and FLUX-1008 are compared on every row in test_gpu_fullsize.py;
# the two larger workloads on their seams plus seeded random rows.
FULL = [("qwen1328", 5, "direct", "fold"), ("qwen1328", 5, "a2a", "partials"), ("wan", 8, "direct", "partials"),
        ("wan", 8, "direct", "fold")]


@pytest.mark.parametrize("name,U,exchange,ring_merge", FULL)
def test_full_size_sampled(name, U, exchange, ring_merge):
    w = synth.WORKLOADS[name]
    q, k, v = w.qkv()
    plan = _plan(w, U, exchange=exchange, ring_merge=ring_merge)
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), out)
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0 and int(plan.range_flag.item()) == 0
    n_random = 64 if name == "wan" else 192
    rows = sample_rows(plan.L, n_random, seed=1)
    ref = _oracle_rows(q, k, v, rows)
    got = f64(out[:, torch.from_numpy(rows)])
    assert_bf16_close(got, ref, name)


@pytest.mark.parametrize("ring_merge", ["fold", "partials"])
def test_padding_never_reaches_outputs(ring_merge):
    """FLUX-1008 (uneven ring blocks 2241/2240): the head-layout buffers are
    filled with NaN before the run, so the padding row of ring block 1 holds
    NaN.  The output must be NaN-free and bit-identical to a clean run."""
    w = synth.WORKLOADS["flux1008"]
    q, k, v = (t.cuda() for t in w.qkv())
    plan = _plan(w, 4, ring_merge=ring_merge)
    clean = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    plan.run(q, k, v, clean)
    for t in (plan.q_h, plan.k_h, plan.v_h, plan.o_h, plan.parts):
        if t is not None:
            t.fill_(float("nan"))
    dirty = torch.empty_like(clean)
    plan.run(q, k, v, dirty)
    torch.cuda.synchronize()
    assert not torch.isnan(dirty).any()
    assert torch.equal(dirty.view(torch.int16), clean.view(torch.int16))


def test_merge_vs_single_shot_on_device():
    """The R-way merge agrees with single-shot attention on the device to
    1e-3 relative RMS (fp32 outputs), FLUX-1008 with R = 2."""
    import sequence_attention_gb300 as sa
    from tests.helpers import MERGE_REL_RMS, rel_rms
    w = synth.WORKLOADS["flux1008"]
    q, k, v = (t.cuda() for t in w.qkv())
    v16 = v.to(torch.float16)
    single = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    sa.dit_attention(q, k, v16, single)
    # keys split in two chunks of one common stride (ring blocks 2241 / 2240)
    L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, 1, 2)
    cap = L.S_cap
    kp = torch.zeros((2, w.B, cap, w.H, w.D), dtype=k.dtype, device="cuda")
    vp = torch.zeros((2, w.B, cap, w.H, w.D), dtype=torch.float16, device="cuda")
    for j in range(2):
        kp[j, :, : L.ring_len[j]] = k[:, L.ring_off[j]:L.ring_off[j] + L.ring_len[j]]
        vp[j, :, : L.ring_len[j]] = v16[:, L.ring_off[j]:L.ring_off[j] + L.ring_len[j]]
    parts = torch.empty((1, 2, w.B, w.S, w.H, w.D), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, 2, w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    sa.dit_attn_partial(q.unsqueeze(0), kp, vp, parts, lse, [w.S], L.ring_len)
    merged = torch.empty((1,) + tuple(q.shape), dtype=torch.float32, device="cuda")
    sa.dit_attn_merge_lse(parts, lse, merged, None, [w.S])
    torch.cuda.synchronize()
    assert rel_rms(f64(merged[0]), f64(single)) <= MERGE_REL_RMS


@pytest.mark.parametrize("B,S,H,U,R,S_txt", [(1, 700, 5, 2, 2, 77), (2, 517, 4, 3, 1, 64)])
def test_double_stream_block_with_rope(B, S, H, U, R, S_txt):
    """Paired text/image streams in, receive preparation with RoPE, ring
    attention, paired streams out, against the oracle's attention over the
    rotated joint sequence (edge-dit.cpp, receive preparation and FLUX
    double-stream blocks)."""
    from oracle import rope as orope
    from sequence_attention_gb300.usp import UspPlan
    D = 128
    qkv = [synth.normal((B, S, H, D), 40 + p, 0.5, "bf16") for p in range(3)]
    cos, sin = synth.rope_tables_joint(S_txt, S, D)
    plan = UspPlan(B, S, H, D, U, R, rope=(cos.cuda(), sin.cuda()))
    txt = [t[:, :S_txt].contiguous().cuda() for t in qkv]
    img = [t[:, S_txt:].contiguous().cuda() for t in qkv]
    out_t = torch.empty((B, S_txt, H, D), dtype=torch.bfloat16, device="cuda")
    out_i = torch.empty((B, S - S_txt, H, D), dtype=torch.bfloat16, device="cuda")
    plan.run_joint(txt, img, out_t, out_i)
    torch.cuda.synchronize()
    c, s = cos.double().numpy(), sin.double().numpy()
    q = orope.rope(f64(qkv[0]), c, s)
    k = orope.rope(f64(qkv[1]), c, s)
    ref, _ = oatt.attention(q, k, f64(qkv[2]))
    got = np.concatenate([f64(out_t), f64(out_i)], axis=1)
    assert_bf16_close(got, ref, "double-stream attention")
    assert int(plan.range_flag.item()) == 0


@pytest.mark.parametrize("U,R", [(2, 2), (1, 3)])
def test_empty_sequence(U, R):
    """S = 0: every call of the step sees zero-size buffers (NULL pointers)
    and launches nothing; the step completes with a clean status."""
    from sequence_attention_gb300.usp import UspPlan
    B, H, D = 1, 3, 64
    q, k, v = (torch.empty((B, 0, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    out = torch.empty((B, 0, H, D), dtype=torch.bfloat16, device="cuda")
    plan = UspPlan(B, 0, H, D, U, R)
    plan.run(q, k, v, out)
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0 and int(plan.range_flag.item()) == 0


def test_half_partials_against_float_partials():
    """The step's default f16 ring partials against f32 ones (both with f32
    output), FLUX-1008-like (R = 2): within the merge bar of 1e-3 rel-RMS.
    (The default step's output against the oracle is covered above.)"""
    from sequence_attention_gb300.usp import UspPlan
    from tests.helpers import MERGE_REL_RMS, rel_rms
    w = synth.WORKLOADS["flux1008"]
    q, k, v = (t.cuda() for t in w.qkv())
    outs = {}
    for pdt in (torch.float16, torch.float32):
        plan = UspPlan(w.B, w.S, w.H, w.D, 4, w.R, out_dtype=torch.float32, parts_dtype=pdt, ring_merge="partials")
        assert plan.parts.dtype == pdt
        outs[pdt] = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.float32, device="cuda")
        plan.run(q, k, v, outs[pdt])
        torch.cuda.synchronize()
        assert int(plan.status.item()) == 0
    assert rel_rms(f64(outs[torch.float16]), f64(outs[torch.float32])) <= MERGE_REL_RMS


@pytest.mark.parametrize("exchange", ["direct", "a2a"])
def test_plan_check_reports_f16_overflow_and_clears(exchange):
    """A V value past f16's range makes the default plan's output non-finite;
    check() raises DIT_ERR_RANGE for it, clears the sticky word, and a plan
    with bf16 V runs the same inputs cleanly."""
    import sequence_attention_gb300 as sa
    from sequence_attention_gb300.usp import UspPlan
    B, S, H, D, U, R = 1, 300, 4, 64, 2, 2
    q = synth.normal((B, S, H, D), 30, 0.5, "bf16").cuda()
    k = synth.normal((B, S, H, D), 31, 0.5, "bf16").cuda()
    v = synth.normal((B, S, H, D), 32, 0.5, "bf16").cuda()
    v[0, 17, 2, 5] = 1.0e6
    out = torch.empty_like(q)
    plan = UspPlan(B, S, H, D, U, R, exchange=exchange)
    plan.run(q, k, v, out)
    with pytest.raises(sa.DitError) as ei:
        plan.check()
    assert ei.value.status == 5
    plan.check()                                  # cleared: no error now
    plan_bf = UspPlan(B, S, H, D, U, R, exchange=exchange, v_dtype=torch.bfloat16)
    plan_bf.run(q, k, v, out, check=True)
    assert torch.isfinite(out.float()).all()
