"""GPU parity of the CFG combine against the oracle.

The kernel evaluates u + g(c - u) in fp32 as fma(g, c - u, u) and rounds
once to the output type; the oracle evaluates it in fp64 and rounds once.
The fp32 evaluation errs by at most |g| |c - u| 2^-24 + half an fp32 ulp, so
the bar is: |gpu - oracle| <= one output ulp of the result plus that fp32
bound (16-bit outputs are then equal almost everywhere), and 1e-5 absolute
for fp32 outputs.  g = 0 and g = 1 are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import cfg as ocfg
from oracle.numeric import to_f64
from tests.helpers import bits

pytestmark = pytest.mark.gpu


def _combine(pred, out_dtype, g):
    import sequence_attention_gb300 as sa
    out = torch.empty(pred.shape[1:], dtype=out_dtype, device="cuda")
    sa.dit_cfg_combine(pred, out, g)
    torch.cuda.synchronize()
    return out


def _ulp_diff(a_bits, b_bits):
    # distance in representable steps, for same-sign finite values
    return np.abs(a_bits.astype(np.int64) - b_bits.astype(np.int64))


@pytest.mark.parametrize("shape,in_dt,out_dt,g", [
    ((2, 1, 256, 4, 64), "f32", "f32", 4.0),        # tiny
    ((2, 4608, 3072), "bf16", "bf16", 3.5),          # FLUX
    ((2, 7145, 3072), "f32", "bf16", 4.0),           # Qwen-Image (fused cast)
    ((2, 999, 37), "bf16", "bf16", 3.5),             # odd length: scalar path
    ((2, 3, 4), "f32", "bf16", 2.0),                 # 8-wide vectors plus a tail of 4
    ((2, 13), "f16", "f32", -1.5),
])
def test_cfg_matches_oracle(shape, in_dt, out_dt, g):
    u = synth.normal(shape[1:], 3, 1.0, in_dt)
    c = synth.normal(shape[1:], 4, 1.0, in_dt)
    pred = torch.stack([u, c]).cuda()
    out = _combine(pred, synth.torch_dtype(out_dt), g)
    ref = ocfg.cfg_combine_bits(bits(pred), in_dt, g, out_dt)
    got = bits(out)
    gv, rv = to_f64(got, out_dt), to_f64(ref, out_dt)
    uu, cc = to_f64(bits(pred[0]), in_dt), to_f64(bits(pred[1]), in_dt)
    ulp = np.spacing(np.abs(rv).astype(np.float32 if out_dt == "f32" else np.float64))
    if out_dt != "f32":
        ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(rv), 2.0 ** -126))[1] - 8 - (3 if out_dt == "f16" else 0))
    fp32_err = abs(g) * np.abs(cc - uu) * 2.0 ** -24 + np.abs(rv) * 2.0 ** -24
    assert np.all(np.abs(gv - rv) <= ulp + fp32_err)
    if out_dt == "f32":
        assert np.max(np.abs(gv - rv)) <= 1e-5
    else:
        assert np.mean(got != ref) < 1e-3


@pytest.mark.parametrize("in_dt", ["bf16", "f32"])
def test_cfg_g0_g1_bit_exact(in_dt):
    shape = (4608, 3072) if in_dt == "bf16" else (1, 256, 4, 64)
    u = synth.normal(shape, 5, 1.0, in_dt)
    c = synth.normal(shape, 6, 1.0, in_dt)
    pred = torch.stack([u, c]).cuda()
    dt = synth.torch_dtype(in_dt)
    assert torch.equal(bits_t(_combine(pred, dt, 0.0)), bits_t(pred[0]))
    assert torch.equal(bits_t(_combine(pred, dt, 1.0)), bits_t(pred[1]))


def bits_t(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def test_cfg_wan_size_samples():
    w = synth.WORKLOADS["wan"]
    pred = w.cfg_pair().cuda()
    out = _combine(pred, torch.bfloat16, w.g)
    idx = np.random.default_rng(0).integers(0, out.numel(), 1 << 16)
    flat_p = pred.view(2, -1)
    sel = torch.from_numpy(idx).cuda()
    pb = bits(torch.stack([flat_p[0, sel], flat_p[1, sel]]))
    ref = ocfg.cfg_combine_bits(pb, "bf16", w.g, "bf16")
    d = _ulp_diff(bits(out.view(-1)[sel]), ref)
    assert d.max() <= 1
