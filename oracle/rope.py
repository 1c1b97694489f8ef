"""Rotary position embedding applied during receive preparation.

Source: edge-dit.cpp "Parallel execution", receive preparation: the CUDA
receive path decodes the all-to-all buffer, extracts the Q/K/V planes, builds
the head-sharded layout and applies RoPE to Q and K; for FLUX double-stream
blocks, paired text and image streams are assembled into the joint attention
sequence.  The pages give no formula.  Reading: the standard rotary embedding
(each pair of head-dim elements rotated by an angle that depends on the
token's position), pairs taken interleaved, (x[2i], x[2i+1]), as FLUX does,
with the angles supplied as cos/sin tables indexed by the token's position in
the joint sequence (text tokens first):

    y[2i]   = x[2i] cos(t, i) - x[2i+1] sin(t, i)
    y[2i+1] = x[2i] sin(t, i) + x[2i+1] cos(t, i)

Evaluated in float64 from the tables' values.
"""
from __future__ import annotations

import numpy as np


def rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """x: [B, S, H, D]; cos, sin: [S, D/2] (angles of token t, pair i)."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(cos, dtype=np.float64)[None, :, None, :]
    s = np.asarray(sin, dtype=np.float64)[None, :, None, :]
    even, odd = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = even * c - odd * s
    y[..., 1::2] = even * s + odd * c
    return y


def joint(txt: np.ndarray, img: np.ndarray) -> np.ndarray:
    """The joint attention sequence of a double-stream block: text tokens
    first, then image tokens, along the sequence axis of [B, S, H, D]."""
    return np.concatenate([np.asarray(txt), np.asarray(img)], axis=1)
