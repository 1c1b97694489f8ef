"""GPU parity of the ring's log-sum-exp merge (dit_attn_merge_lse) against the
oracle's merge (SGLang Diffusion "Parallelism Overview", What happens to the
shapes and Constraints: ranks of a ring group hold the same heads over
different rows, and their partials fold with the online-softmax merge).

The kernel evaluates the merge in fp32 (one accurate exp per part for the
sum, one log, one exp per part for the weights, an FMA chain over the parts)
and rounds once to the output type.  Against the fp64 oracle on the same
partial values the error is then a few fp32 ulps of the result's scale plus,
for a 16-bit output, half an ulp of that type:
    |got - ref| <= 1e-5 * max_j |O_j| + half_ulp(ref, out type)
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from tests.helpers import DT_NAME, f64, half_ulp

pytestmark = pytest.mark.gpu


def _merge_case(n_q, n, B, S, H, D, pdt, odt, seed, pad_heads=0, lse_out=True):
    import sequence_attention_gb300 as sa
    rng = np.random.default_rng(seed)
    Hs = H + pad_heads                                  # storage heads (a strided view of H)
    parts_full = torch.from_numpy(rng.standard_normal((n_q, n, B, S, Hs, D)).astype(np.float32)).to(pdt)
    lse_full = torch.from_numpy((rng.standard_normal((n_q, n, B, Hs, S)) * 4).astype(np.float32))
    q_len = [S - 3 * r for r in range(n_q)]
    # an all-empty row and one empty chunk
    lse_full[:, :, :, :, 2] = -math.inf
    parts_full[:, :, :, 2] = 0
    lse_full[0, n - 1, :, :, 4] = -math.inf
    out = torch.full((n_q, B, S, Hs, D), float("nan"), dtype=odt, device="cuda")
    lo = torch.full((n_q, B, Hs, S), float("nan"), dtype=torch.float32, device="cuda") if lse_out else None
    pc, lc = parts_full.cuda(), lse_full.cuda()
    sa.dit_attn_merge_lse(pc[..., :H, :], lc[:, :, :, :H, :], out[..., :H, :],
                          None if lo is None else lo[:, :, :H, :], q_len)
    torch.cuda.synchronize()
    scale = float(parts_full.float().abs().max())
    for r in range(n_q):
        rows = q_len[r]
        o_ref, l_ref = oatt.merge([(f64(parts_full[r, j, :, :rows, :H]), f64(lse_full[r, j, :, :H, :rows]))
                                   for j in range(n)])
        got = f64(out[r, :, :rows, :H])
        bound = 1e-5 * scale + (half_ulp(o_ref, DT_NAME[odt]) if odt != torch.float32 else 0.0)
        err = np.abs(got - o_ref)
        assert np.all(err <= bound), f"merge r={r}: max excess {np.max(err - bound):.3e}"
        # rows past the block, and padded heads, are not written
        assert torch.isnan(out[r, :, rows:].float()).all()
        assert torch.isnan(out[r, ..., H:, :].float()).all()
        if lo is not None:
            gl = f64(lo[r, :, :H, :rows])
            fin = np.isfinite(l_ref)
            assert np.array_equal(np.isneginf(gl), np.isneginf(l_ref))
            assert np.max(np.abs(gl[fin] - l_ref[fin]), initial=0.0) <= 1e-5 * max(1.0, np.abs(l_ref[fin]).max())
            assert torch.isnan(lo[r, :, :, rows:]).all() and torch.isnan(lo[r, :, H:]).all()


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("pdt", [torch.float32, torch.float16, torch.bfloat16])
def test_merge_every_part_count(n, pdt):
    _merge_case(2, n, 2, 131, 3, 64, pdt, torch.float32, seed=n, pad_heads=1)


@pytest.mark.parametrize("odt", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [8, 24, 128])
def test_merge_output_types_and_head_dims(odt, D):
    """D = 8 and 24 (three 8-element chunks per head: not a power of two)
    take the same kernel as the workloads' D = 128."""
    _merge_case(3, 2, 1, 77, 5, D, torch.float16, odt, seed=D, pad_heads=2, lse_out=(D != 24))


def test_merge_flux1008_shape():
    """The step's merge at FLUX-1008 size: R = 2 ring blocks of 2241/2240
    rows, 24 heads, f16 partials, bf16 output (the launch the bench times)."""
    import sequence_attention_gb300 as sa
    w = synth.WORKLOADS["flux1008"]
    L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, 4, w.R)
    R, cap = w.R, L.S_cap
    rng = np.random.default_rng(11)
    parts = torch.from_numpy(rng.standard_normal((R, R, w.B, cap, w.H, w.D)).astype(np.float32)).half()
    lse = torch.from_numpy((rng.standard_normal((R, R, w.B, w.H, cap)) * 2).astype(np.float32))
    out = torch.empty((R, w.B, cap, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    sa.dit_attn_merge_lse(parts.cuda(), lse.cuda(), out, None, L.ring_real)
    torch.cuda.synchronize()
    scale = float(parts.float().abs().max())
    for r in range(R):
        rows = L.ring_real[r]
        o_ref, _ = oatt.merge([(f64(parts[r, j, :, :rows]), f64(lse[r, j, :, :, :rows])) for j in range(R)])
        err = np.abs(f64(out[r, :, :rows]) - o_ref)
        assert np.all(err <= 1e-5 * scale + half_ulp(o_ref, "bf16"))


def test_merge_wan_shape_sampled():
    """Wan-like R = 4 merge at full size (18900 rows per block, 40 heads,
    f16 partials), checked on seeded rows of every block including the first
    and last ones."""
    import sequence_attention_gb300 as sa
    w = synth.WORKLOADS["wan"]
    L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, 8, w.R)
    R, cap = w.R, L.S_cap
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    parts = torch.randn((R, R, w.B, cap, w.H, w.D), generator=g, device="cuda").half()
    lse = torch.randn((R, R, w.B, w.H, cap), generator=g, device="cuda") * 3
    out = torch.empty((R, w.B, cap, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    sa.dit_attn_merge_lse(parts, lse, out, None, L.ring_real)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    scale = float(parts.float().abs().max())
    for r in range(R):
        rows = np.unique(np.concatenate([[0, cap - 1], rng.integers(0, cap, 200)]))
        sel = torch.from_numpy(rows).cuda()
        o_ref, _ = oatt.merge([(f64(parts[r, j][:, sel]), f64(lse[r, j][:, :, sel])) for j in range(R)])
        err = np.abs(f64(out[r][:, sel]) - o_ref)
        assert np.all(err <= 1e-5 * scale + half_ulp(o_ref, "bf16"))
