"""Classifier-free guidance combine.

Source: edge-dit.cpp "Parallel execution", classifier-free guidance: the
unconditional and conditional predictions are combined as
p_cfg = p_uncond + guidance_scale * (p_cond - p_uncond); under CFG
parallelism rank 0 runs the unconditional branch and rank 1 the conditional
one, so a stacked [2, ...] tensor holds index 0 = uncond, 1 = cond.

The combine is evaluated literally in float64 and rounded once to the output
storage type (round to nearest even).
"""
from __future__ import annotations

import numpy as np

from .numeric import from_f64, to_f64


def cfg_combine_f64(p_uncond: np.ndarray, p_cond: np.ndarray, g: float) -> np.ndarray:
    u = np.asarray(p_uncond, dtype=np.float64)
    c = np.asarray(p_cond, dtype=np.float64)
    return u + float(g) * (c - u)


def cfg_combine_bits(pred_bits: np.ndarray, in_dt: str, g: float, out_dt: str) -> np.ndarray:
    """pred_bits: stacked [2, ...] storage bits (0 = uncond, 1 = cond)."""
    u = to_f64(pred_bits[0], in_dt)
    c = to_f64(pred_bits[1], in_dt)
    return from_f64(cfg_combine_f64(u, c, g), out_dt)
