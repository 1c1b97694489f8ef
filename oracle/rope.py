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


def receive_prep(L, recv: np.ndarray, wire_dt: str, dst_dts, cos: np.ndarray, sin: np.ndarray,
                 rope_planes: int):
    """Head-sharded planes of every rank from the received buffers, with the
    rotary embedding applied to the planes whose bit is set in rope_planes.

    Returns {(r, v): [plane_0, ...]} with planes of shape [B, S_r, Hl, D]:
    a rotated plane as float64 (the exact rotation of the received values,
    before the rounding to its destination type); any other plane as the
    storage bits of dst_dts[p], as ``ulysses.s2h_unpack`` gives them.  Row s
    of ring block r is the token at joint position ring_off[r] + s; rows of
    an lcm(SP, 64)-padded layout at or past S are padding, never rotated
    (xLLM "DiT Architecture and Capability Matrix": the padding is not part
    of the sequence).
    """
    from . import numeric, ulysses

    kinds = [wire_dt if (rope_planes >> p) & 1 else dt for p, dt in enumerate(dst_dts)]
    ranks = ulysses.s2h_unpack(L, recv, wire_dt, kinds)
    for (r, _v), planes in ranks.items():
        # the tables hold the S real tokens: rows of a padded layout at or
        # past S (sequence padding) are not rotated and stay zero
        n = L.real_rows(r)
        rows = slice(L.ring_off[r], L.ring_off[r] + n)
        for p in range(len(planes)):
            if (rope_planes >> p) & 1:
                x = numeric.to_f64(planes[p], wire_dt)
                x[:, :n] = rope(x[:, :n], np.asarray(cos)[rows], np.asarray(sin)[rows])
                planes[p] = x
    return ranks
