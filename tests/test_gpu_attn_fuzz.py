"""Seeded random attention partials on the tensor cores against the fp64
oracle.  Batches up to 3, up to 5 heads, D 64 or 128, 1-3 query blocks and
1-4 key blocks of random lengths (empty and single-row blocks included),
bf16 or f16 Q/K, f16 or bf16 V, f32, bf16 or f16 output.  Rows past each
block's length hold NaN in every input and output buffer: they must be
neither read nor written."""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from tests.helpers import LSE_ABS, assert_bf16_close, f64, max_abs

pytestmark = pytest.mark.gpu

_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _lengths(rng, n):
    out = []
    for _ in range(n):
        u = rng.random()
        out.append(0 if u < 0.1 else 1 if u < 0.2 else int(rng.integers(2, 400)))
    return out


@pytest.mark.parametrize("seed", range(16))
def test_random_partials(seed):
    import sequence_attention_gb300 as sa
    rng = np.random.default_rng(700 + seed)
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 6))
    D = int(rng.choice([64, 128]))
    n_q, n_kv = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    q_len, kv_len = _lengths(rng, n_q), _lengths(rng, n_kv)
    if max(q_len) == 0:
        q_len[0] = 77
    qk_dt, v_dt = str(rng.choice(["bf16", "f16"])), str(rng.choice(["f16", "bf16"]))
    o_dt = str(rng.choice(["f32", "bf16", "f16"]))
    Sq, Sk = max(q_len), max(max(kv_len), 1)
    q = synth.normal((n_q, B, Sq, H, D), seed, 0.5, "f32")
    k = synth.normal((n_kv, B, Sk, H, D), seed + 1, 0.5, "f32")
    v = synth.normal((n_kv, B, Sk, H, D), seed + 2, 0.5, "f32")
    q, k, v = q.to(_DT[qk_dt]), k.to(_DT[qk_dt]), v.to(_DT[v_dt])
    for r, L in enumerate(q_len):
        q[r, :, L:] = float("nan")
    for j, L in enumerate(kv_len):
        k[j, :, L:] = float("nan")
        v[j, :, L:] = float("nan")
    o = torch.full((n_q, n_kv, B, Sq, H, D), float("nan"), dtype=_DT[o_dt], device="cuda")
    lse = torch.full((n_q, n_kv, B, H, Sq), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_attn_partial(q.cuda(), k.cuda(), v.cuda(), o, lse, q_len, kv_len, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    what = f"B{B} H{H} D{D} q{q_len} kv{kv_len} {qk_dt}/{v_dt}->{o_dt}"
    for r, Lq in enumerate(q_len):
        for j, Lk in enumerate(kv_len):
            got_o, got_l = o[r, j].cpu(), lse[r, j].cpu()
            assert torch.isnan(got_o[:, Lq:]).all() and torch.isnan(got_l[:, :, Lq:]).all(), what
            if Lq == 0:
                continue
            go, gl = f64(got_o[:, :Lq]), f64(got_l[:, :, :Lq])
            if Lk == 0:
                assert np.all(go == 0) and np.all(np.isneginf(gl)), what
                continue
            o_ref, l_ref = oatt.partial(f64(q[r, :, :Lq]), f64(k[j, :, :Lk]), f64(v[j, :, :Lk]), Lk)
            assert_bf16_close(go, o_ref, f"{what} pair ({r},{j})")
            assert max_abs(gl, l_ref) <= LSE_ABS, what


def _segment_lengths(rng, n):
    """Zero, one, tile-boundary (127..129, 255..257) and random lengths."""
    special = [0, 1, 127, 128, 129, 255, 256, 257]
    return [int(rng.choice(special)) if rng.random() < 0.4 else int(rng.integers(2, 500)) for _ in range(n)]


@pytest.mark.parametrize("seed", range(12))
def test_random_varlen(seed):
    """Packed variable-length attention: 1-20 sequences (more than one launch
    of 8), query and key segments of independent lengths (empty ones
    included), packing that starts past row 0, rows outside every sequence
    (NaN, never written), random types and D."""
    import sequence_attention_gb300 as sa
    rng = np.random.default_rng(1300 + seed)
    n = int(rng.integers(1, 21))
    H, D = int(rng.integers(1, 5)), int(rng.choice([64, 128]))
    qk_dt, v_dt = str(rng.choice(["bf16", "f16"])), str(rng.choice(["f16", "bf16"]))
    o_dt = str(rng.choice(["f32", "bf16", "f16"]))
    lq, lk = _segment_lengths(rng, n), _segment_lengths(rng, n)
    q0, k0 = int(rng.integers(0, 40)), int(rng.integers(0, 40))
    cu_q, cu_k = list(np.cumsum([q0] + lq)), list(np.cumsum([k0] + lk))
    cu_q, cu_k = [int(x) for x in cu_q], [int(x) for x in cu_k]
    Tq, Tk = cu_q[-1] + int(rng.integers(0, 9)), max(cu_k[-1] + int(rng.integers(0, 9)), 1)
    q = synth.normal((Tq, H, D), 40 * seed, 0.5, "f32").to(_DT[qk_dt])
    k = synth.normal((Tk, H, D), 40 * seed + 1, 0.5, "f32").to(_DT[qk_dt])
    v = synth.normal((Tk, H, D), 40 * seed + 2, 0.5, "f32").to(_DT[v_dt])
    o = torch.full((Tq, H, D), float("nan"), dtype=_DT[o_dt], device="cuda")
    lse = torch.full((H, Tq), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa.dit_attn_varlen(q.cuda(), k.cuda(), v.cuda(), o, cu_q, cu_k, lse, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    what = f"n{n} H{H} D{D} lq{lq} lk{lk} start {q0}/{k0} {qk_dt}/{v_dt}->{o_dt}"
    ref, lref = oatt.varlen(f64(q), f64(k), f64(v), cu_q, cu_k)
    got, gl = f64(o), lse.cpu().double().numpy()
    inside = np.zeros(Tq, bool)
    for s in range(n):
        rows = slice(cu_q[s], cu_q[s + 1])
        inside[rows] = True
        if lq[s] == 0:
            continue
        if lk[s] == 0:
            assert np.all(got[rows] == 0) and np.all(np.isneginf(gl[:, rows])), what
            continue
        assert_bf16_close(got[rows], ref[rows], f"{what} segment {s}")
        assert max_abs(gl[:, rows], lref[:, rows]) <= LSE_ABS, what
    assert np.all(np.isnan(got[~inside])) and np.all(np.isnan(gl[:, ~inside])), what
