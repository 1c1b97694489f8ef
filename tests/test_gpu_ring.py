"""GPU parity of the folded ring attention (dit_attn_ring) against the oracle.

Each query block attends every key/value block of the ring in turn and the
kernel folds each block into one running result with the online softmax
(SGLang Diffusion "Parallelism Overview", What happens to the shapes and
Constraints: Q stays while the K/V chunks visit, each hop merged by the
online softmax).  The result must be the oracle's attention over the
concatenated valid keys of all blocks: the tensor-core path at the bf16 bars
(max-abs 2e-2, rel-RMS 5e-3; log-sum-exp within 1e-4), the fp32 path within
1e-5, and against the device's own partials + R-way merge within the merge
bar (1e-3 rel-RMS, fp32 outputs).
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from tests.helpers import F32_MAX_ABS, LSE_ABS, MERGE_REL_RMS, assert_bf16_close, bits, f64, max_abs, rel_rms

pytestmark = pytest.mark.gpu


def _blocks(x, lens, cap):
    """[B, sum(lens), H, D] -> [n, B, cap, H, D] blocks, NaN past each length."""
    B, _, H, D = x.shape
    out = torch.full((len(lens), B, cap, H, D), float("nan"), dtype=x.dtype)
    off = 0
    for j, L in enumerate(lens):
        out[j, :, :L] = x[:, off:off + L]
        off += L
    return out


def _ring(q, k, v, q_lens, kv_lens, v_dt, o_dt, Hs, with_lse=True):
    """Run dit_attn_ring on padded block tensors with Hs >= H storage heads;
    returns (o [n_q, B, cap, Hs, D] on the host, lse or None)."""
    import sequence_attention_gb300 as sa
    B, _, H, D = q.shape
    cq, ck = max(max(q_lens), 1), max(max(kv_lens), 1)
    qb, kb, vb = _blocks(q, q_lens, cq), _blocks(k, kv_lens, ck), _blocks(v.to(v_dt), kv_lens, ck)
    def store(x):
        full = torch.zeros(x.shape[:3] + (Hs, D), dtype=x.dtype)
        full[..., :H, :] = x
        return full.cuda()
    qd, kd, vd = store(qb), store(kb), store(vb)
    o = torch.full((len(q_lens), B, cq, Hs, D), float("nan"), dtype=o_dt, device="cuda")
    lse = torch.full((len(q_lens), B, Hs, cq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_attn_ring(qd[..., :H, :], kd[..., :H, :], vd[..., :H, :], o[..., :H, :],
                     None if lse is None else lse[:, :, :H, :], q_lens, kv_lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o.cpu(), (None if lse is None else lse.cpu())


CASES = [
    # B, H, D, q block lengths, key block lengths
    (1, 2, 128, [300], [200, 133]),
    (2, 3, 128, [190, 190], [128, 0, 77]),              # an empty middle block
    (1, 1, 128, [2241, 2240], [2241, 2240]),            # FLUX-1008's ring blocks, one head
    (1, 2, 64, [640, 5], [1000, 1000, 1000, 997]),      # D = 64, four blocks, a 5-row query block
    (1, 1, 128, [129], [1, 0, 0, 127]),                  # one-key block, empty blocks
    (2, 2, 128, [257], [8300, 100]),                     # a long 65-tile block
    (1, 2, 128, [100], [0, 0]),                          # every key block empty
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("v_dt,o_dt", [(torch.float16, torch.bfloat16), (torch.float16, torch.float32),
                                       (torch.bfloat16, torch.float16)])
def test_ring_matches_oracle(case, v_dt, o_dt):
    B, H, D, q_lens, kv_lens = case
    Sq, Sk = sum(q_lens), sum(kv_lens)
    q = synth.normal((B, Sq, H, D), 90, 0.5, "bf16")
    k = synth.normal((B, max(Sk, 1), H, D), 91, 0.5, "bf16")[:, :Sk]
    v = synth.normal((B, max(Sk, 1), H, D), 92, 0.5, "bf16")[:, :Sk]
    Hs = H + 1                                           # one padded head the kernel must not touch
    o, lse = _ring(q, k, v, q_lens, kv_lens, v_dt, o_dt, Hs)
    vq = v.to(v_dt)
    o_ref, l_ref = oatt.attention(f64(q), f64(k), f64(vq))
    off = 0
    for r, L in enumerate(q_lens):
        got = f64(o[r, :, :L, :H])
        if Sk == 0:
            assert np.all(got == 0) and np.all(np.isneginf(f64(lse[r, :, :H, :L])))
        else:
            assert_bf16_close(got, o_ref[:, off:off + L], f"query block {r}")
            assert max_abs(f64(lse[r, :, :H, :L]), l_ref[:, :, off:off + L]) <= LSE_ABS
        # rows past the block and the padded head are never written
        assert torch.isnan(o[r, :, L:].float()).all() and torch.isnan(o[r, ..., H:, :].float()).all()
        assert torch.isnan(lse[r, :, H:]).all() and torch.isnan(lse[r, :, :, L:]).all()
        off += L


@pytest.mark.parametrize("case", CASES[:4])
def test_ring_fp32_path(case):
    B, H, D, q_lens, kv_lens = case
    D = 64 if D == 128 else D
    Sq, Sk = sum(q_lens), sum(kv_lens)
    q = synth.normal((B, Sq, H, D), 93, 1.0, "f32")
    k = synth.normal((B, Sk, H, D), 94, 1.0, "f32")
    v = synth.normal((B, Sk, H, D), 95, 1.0, "f32")
    o, lse = _ring(q, k, v, q_lens, kv_lens, torch.float32, torch.float32, H)
    o_ref, l_ref = oatt.attention(f64(q), f64(k), f64(v))
    off = 0
    for r, L in enumerate(q_lens):
        assert max_abs(f64(o[r, :, :L]), o_ref[:, off:off + L]) <= F32_MAX_ABS
        assert max_abs(f64(lse[r, :, :, :L]), l_ref[:, :, off:off + L]) <= F32_MAX_ABS
        off += L


def test_ring_equals_partials_and_merge_on_device():
    """Folding in the kernel and merging written partials agree within the
    merge bar (FLUX-1008-like R = 2 ring blocks, all 24 heads, fp32 outputs)."""
    import sequence_attention_gb300 as sa
    w = synth.WORKLOADS["flux1008"]
    L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, 1, w.R)
    q, k, v = w.qkv()
    rl, cap = L.ring_real, L.S_cap
    qb = _blocks(q, rl, cap).cuda()
    kb = _blocks(k, rl, cap).cuda()
    vb = _blocks(v.to(torch.float16), rl, cap).cuda()
    ring = torch.empty((w.R, w.B, cap, w.H, w.D), dtype=torch.float32, device="cuda")
    sa.dit_attn_ring(qb, kb, vb, ring, None, rl, rl)
    parts = torch.empty((w.R, w.R, w.B, cap, w.H, w.D), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.R, w.R, w.B, w.H, cap), dtype=torch.float32, device="cuda")
    sa.dit_attn_partial(qb, kb, vb, parts, lse, rl, rl)
    merged = torch.empty_like(ring)
    sa.dit_attn_merge_lse(parts, lse, merged, None, rl)
    torch.cuda.synchronize()
    for r in range(w.R):
        n = rl[r]
        assert rel_rms(f64(ring[r, :, :n]), f64(merged[r, :, :n])) <= MERGE_REL_RMS


def test_ring_argument_checks():
    import sequence_attention_gb300 as sa
    q = torch.zeros((2, 1, 64, 2, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((2, 1, 64, 2, 128), dtype=torch.float16, device="cuda")
    o = torch.zeros((2, 1, 64, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa.DitError):
        sa.dit_attn_ring(q, q, v, o, None, [64, 64], [64, 64], scale=-1.0)       # scale must be positive
    with pytest.raises(sa.DitError):
        sa.dit_attn_ring(q, q, v, o, None, [64, -1], [64, 64])                   # negative length
    with pytest.raises(sa.DitError):
        sa.dit_attn_ring(q, q, v, o.expand(2, 1, 64, 2, 128).as_strided(o.shape, (0,) + o.stride()[1:]), None,
                         [64, 64], [64, 64])                                       # two blocks on one address


@pytest.mark.parametrize("v_dt,o_dt", [(torch.float16, torch.bfloat16), (torch.float32, torch.float32)])
def test_ring_rows_into_one_sequence_tensor(v_dt, o_dt):
    """dit_attn_ring_rows places query block r at rows o_row0[r] of one
    [B,S,H,D] tensor: bit for bit what dit_attn_ring writes per block, every
    row written once, nothing else touched (an empty block in the middle)."""
    import sequence_attention_gb300 as sa
    B, H, D = 2, 3, 64
    q_lens, kv_lens = [130, 0, 77, 201], [130, 64, 77, 201]
    f32 = v_dt == torch.float32
    kind = "f32" if f32 else "bf16"
    Sq, Sk = sum(q_lens), sum(kv_lens)
    q = synth.normal((B, Sq, H, D), 96, 0.5, kind)
    k = synth.normal((B, Sk, H, D), 97, 0.5, kind)
    v = synth.normal((B, Sk, H, D), 98, 0.5, kind)
    cq, ck = max(q_lens), max(kv_lens)
    qd, kd, vd = (_blocks(x, l, c).cuda() for x, l, c in ((q, q_lens, cq), (k, kv_lens, ck), (v.to(v_dt), kv_lens, ck)))
    # per-block outputs, then the same into one tensor with a spare row at the end
    ref = torch.full((len(q_lens), B, cq, H, D), float("nan"), dtype=o_dt, device="cuda")
    sa.dit_attn_ring(qd, kd, vd, ref, None, q_lens, kv_lens)
    out = torch.full((B, Sq + 1, H, D), float("nan"), dtype=o_dt, device="cuda")
    row0 = [sum(q_lens[:r]) for r in range(len(q_lens))]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_attn_ring_rows(qd, kd, vd, out, row0, None, q_lens, kv_lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for r, L in enumerate(q_lens):
        np.testing.assert_array_equal(bits(out[:, row0[r]:row0[r] + L]), bits(ref[r, :, :L]))
    assert torch.isnan(out[:, Sq:].float()).all()                    # the spare row is untouched
    assert not torch.isnan(out[:, :Sq].float()).any()
    if not f32:
        o_ref, _ = oatt.attention(f64(q), f64(k), f64(v.to(v_dt)))
        # every query row attends every key of every block: the full attention
        assert_bf16_close(f64(out[:, :Sq]), o_ref, "ring rows")


def test_ring_rows_argument_checks():
    import sequence_attention_gb300 as sa
    q = torch.zeros((2, 1, 64, 2, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((2, 1, 64, 2, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros((1, 128, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa.DitError):
        sa.dit_attn_ring_rows(q, q, v, out, [0, 32], None, [64, 64], [64, 64])    # blocks' rows overlap
    with pytest.raises(sa.DitError):
        sa.dit_attn_ring_rows(q, q, v, out, [0, -1], None, [64, 64], [64, 64])    # negative row
    sa.dit_attn_ring_rows(q, q, v, out, [64, 0], None, [64, 64], [64, 64])        # any order of disjoint rows
    torch.cuda.synchronize()


@pytest.mark.parametrize("seed", range(6))
def test_ring_rows_fuzz(seed):
    """Random block counts and lengths (empty blocks included), output rows
    placed with random gaps between the blocks in one tensor: every block's
    rows are what dit_attn_ring writes for it, and the gaps stay untouched."""
    import sequence_attention_gb300 as sa
    rng = np.random.default_rng(1000 + seed)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    D = int(rng.choice([64, 128]))
    n_q, n_kv = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    q_lens = [int(x) for x in rng.integers(0, 300, size=n_q)]
    kv_lens = [int(x) for x in rng.integers(0, 400, size=n_kv)]
    if sum(q_lens) == 0:
        q_lens[0] = 1
    gaps = [int(x) for x in rng.integers(0, 5, size=n_q + 1)]
    row0, at = [], gaps[0]
    for r in range(n_q):
        row0.append(at)
        at += q_lens[r] + gaps[r + 1]
    cq, ck = max(max(q_lens), 1), max(max(kv_lens), 1)
    q = synth.normal((n_q, B, cq, H, D), 2000 + seed, 0.5, "bf16").cuda()
    k = synth.normal((n_kv, B, ck, H, D), 3000 + seed, 0.5, "bf16").cuda()
    v = synth.normal((n_kv, B, ck, H, D), 4000 + seed, 0.5, "f16").cuda()
    ref = torch.full((n_q, B, cq, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    sa.dit_attn_ring(q, k, v, ref, None, q_lens, kv_lens)
    out = torch.full((B, at, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    sa.dit_attn_ring_rows(q, k, v, out, row0, None, q_lens, kv_lens)
    torch.cuda.synchronize()
    written = torch.zeros(at, dtype=torch.bool)
    for r in range(n_q):
        L = q_lens[r]
        np.testing.assert_array_equal(bits(out[:, row0[r]:row0[r] + L]), bits(ref[r, :, :L]))
        written[row0[r]:row0[r] + L] = True
    assert torch.isnan(out[:, ~written.cuda()].float()).all()
