"""Seeded random configurations of the whole hot path through UspPlan: the
Ulysses and ring degrees, uneven splits, head padding or none, lcm(U*R, 64)
sequence padding, RoPE receive preparation and the e4m3 wire for Q and V
drawn at random.  The output is compared in full with the fp64 oracle's
attention over the same (rotated, e4m3-decoded where the wire is e4m3)
inputs, at the bf16 bars."""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import fp8 as ofp8
from oracle import rope as orope
from tests.helpers import assert_bf16_close, f64

pytestmark = pytest.mark.gpu


def _decoded(x):
    return ofp8.dequantize_heads(*ofp8.quantize_heads(x.astype(np.float32))).astype(np.float64)


@pytest.mark.parametrize("seed", range(12))
def test_random_usp_configuration(seed):
    from sequence_attention_gb300.usp import UspPlan
    rng = np.random.default_rng(900 + seed)
    U, R = int(rng.integers(1, 5)), int(rng.integers(1, 4))
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 7))
    D = int(rng.choice([64, 128]))
    S = int(rng.integers(U * R, 700))
    pad_heads, pad_lcm64 = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    use_rope, fp8_qv = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    q, k, v = (synth.normal((B, S, H, D), 50 * seed + p, 0.5, "bf16") for p in range(3))
    rope = None
    if use_rope:
        cos, sin = synth.rope_tables_linear(S, D)
        rope = (cos.cuda(), sin.cuda())
    plan = UspPlan(B, S, H, D, U, R, rope=rope, fp8_qv=fp8_qv, pad_heads=pad_heads, pad_lcm64=pad_lcm64)
    out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), out)
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0
    qr, kr, vr = f64(q), f64(k), f64(v)
    if fp8_qv:
        qr, vr = _decoded(qr), _decoded(vr)
    if use_rope:
        c, s = cos.double().numpy(), sin.double().numpy()
        qr, kr = orope.rope(qr, c, s), orope.rope(kr, c, s)
    ref, _ = oatt.attention(qr, kr, vr)
    assert_bf16_close(f64(out), ref, f"B{B} S{S} H{H} D{D} U{U} R{R} pad_heads={pad_heads} "
                                     f"lcm64={pad_lcm64} rope={use_rope} e4m3={fp8_qv}")


@pytest.mark.parametrize("B,S,H,D,U,R", [(1, 1000, 2, 128, 1, 8), (2, 601, 3, 64, 2, 8), (1, 900, 16, 64, 8, 8)])
def test_eight_ring_blocks(B, S, H, D, U, R):
    """The largest ring (8 blocks, 64 (query, key) partials per head walked
    by the kernel that visits every key block) and 64 virtual ranks, end to
    end against the oracle."""
    from sequence_attention_gb300.usp import UspPlan
    q, k, v = (synth.normal((B, S, H, D), 70 + p, 0.5, "bf16") for p in range(3))
    plan = UspPlan(B, S, H, D, U, R)
    out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    plan.run(q.cuda(), k.cuda(), v.cuda(), out)
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0
    ref, _ = oatt.attention(f64(q), f64(k), f64(v))
    assert_bf16_close(f64(out), ref, f"B{B} S{S} H{H} D{D} U{U} R{R}")


@pytest.mark.parametrize("seed", range(10))
def test_random_joint_step(seed):
    """The double-stream step (paired text and image tensors in, the two
    output streams written back) on random configurations: the text length
    0, S or anything between, with the degrees, layout flags, RoPE and the
    e4m3 wire drawn as in the step fuzz.  The two outputs, side by side,
    must be the oracle's attention over the joint sequence."""
    from sequence_attention_gb300.usp import UspPlan
    rng = np.random.default_rng(1500 + seed)
    U, R = int(rng.integers(1, 5)), int(rng.integers(1, 4))
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 7))
    D = int(rng.choice([64, 128]))
    S = int(rng.integers(U * R, 700))
    pad_heads, pad_lcm64 = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    use_rope, fp8_qv = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    u = rng.random()
    S_txt = 0 if u < 0.2 else S if u < 0.4 else int(rng.integers(1, S))
    q, k, v = (synth.normal((B, S, H, D), 50 * seed + 7 + p, 0.5, "bf16") for p in range(3))
    rope = None
    if use_rope:
        cos, sin = synth.rope_tables_linear(S, D)
        rope = (cos.cuda(), sin.cuda())
    plan = UspPlan(B, S, H, D, U, R, rope=rope, fp8_qv=fp8_qv, pad_heads=pad_heads, pad_lcm64=pad_lcm64)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    txt = tuple(x[:, :S_txt].contiguous() for x in (qd, kd, vd)) if S_txt > 0 else None
    img = tuple(x[:, S_txt:].contiguous() for x in (qd, kd, vd)) if S_txt < S else None
    out_t = torch.full((B, S_txt, H, D), float("nan"), dtype=torch.bfloat16, device="cuda") if S_txt else None
    out_i = torch.full((B, S - S_txt, H, D), float("nan"), dtype=torch.bfloat16, device="cuda") \
        if S_txt < S else None
    plan.run_joint(txt, img, out_t, out_i)
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0
    got = torch.cat([t for t in (out_t, out_i) if t is not None], dim=1)
    qr, kr, vr = f64(q), f64(k), f64(v)
    if fp8_qv:
        qr, vr = _decoded(qr), _decoded(vr)
    if use_rope:
        c, s = cos.double().numpy(), sin.double().numpy()
        qr, kr = orope.rope(qr, c, s), orope.rope(kr, c, s)
    ref, _ = oatt.attention(qr, kr, vr)
    assert_bf16_close(f64(got), ref, f"B{B} S{S} S_txt{S_txt} H{H} D{D} U{U} R{R} pad_heads={pad_heads} "
                                     f"lcm64={pad_lcm64} rope={use_rope} e4m3={fp8_qv}")
