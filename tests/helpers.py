"""Shared helpers of the GPU parity tests (comparison metrics, conversions)."""
from __future__ import annotations

import math

import numpy as np
import torch

# Parity bars (tensor-core bf16 path vs the fp64 oracle; fp32 path; GPU
# R-way merge vs GPU single shot).
BF16_MAX_ABS = 2e-2
BF16_REL_RMS = 5e-3
F32_MAX_ABS = 1e-5
MERGE_REL_RMS = 1e-3
LSE_ABS = 1e-4


def rel_rms(x, y) -> float:
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    den = math.sqrt(float(np.sum(y * y)))
    return math.sqrt(float(np.sum((x - y) ** 2))) / (den if den > 0 else 1.0)


def max_abs(x, y) -> float:
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(y, np.float64)))) if np.size(x) else 0.0


def assert_bf16_close(gpu, ref, what=""):
    ma, rr = max_abs(gpu, ref), rel_rms(gpu, ref)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    assert ma <= BF16_MAX_ABS and rr <= BF16_REL_RMS, f"{what}: max-abs {ma:.3e}, rel-RMS {rr:.3e}"
    return ma, rr


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().to("cpu").contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.int32).numpy().view(np.uint32)


DT_NAME = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


def sample_rows(L, n_random: int, seed: int = 0):
    """Query rows to check at full size: first/last row of every virtual rank
    and ring block (the UAA and ring seams) plus seeded random rows."""
    rows = set()
    for off, n in zip(L.rank_off, L.rank_len):
        if n:
            rows.update((off, off + n - 1))
    rng = np.random.default_rng(seed)
    rows.update(int(x) for x in rng.integers(0, L.S, n_random))
    return np.array(sorted(rows))


_PRECISION = {"bf16": (8, -133), "f16": (11, -24), "f32": (24, -149)}


def half_ulp(y, dt: str) -> np.ndarray:
    """Half a unit in the last place of |y|'s binade in type dt (subnormal
    spacing at the bottom): the largest error of a round-to-nearest."""
    p, sub = _PRECISION[dt]
    a = np.abs(np.asarray(y, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return 0.5 * np.exp2(np.maximum(e - (p - 1), sub))


def assert_rotation_close(gpu, exact, x, dt: str, what=""):
    """A pair rotation done in fp32 (one rounded product, one fused
    multiply-add) then rounded to dt: the error is at most 2^-23 (|x0| + |x1|)
    before the final rounding plus half an ulp of dt.  x are the rotated
    inputs, [..., D]."""
    gpu = np.asarray(gpu, dtype=np.float64)
    exact = np.asarray(exact, dtype=np.float64)
    m = np.abs(x[..., 0::2]) + np.abs(x[..., 1::2])
    m = np.repeat(m, 2, axis=-1)
    bound = 2.0 ** -23 * m + half_ulp(np.maximum(np.abs(gpu), np.abs(exact)), dt)
    err = np.abs(gpu - exact)
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} beyond the bound, worst {err[bad].max():.3e}"
