"""Unified sequence parallelism (Ulysses inside, ring outside), end to end.

Sources:
* SGLang Diffusion "Parallelism Overview", "What happens to the shapes":
  [B, S/(U*R), H, D] -> Ulysses all-to-all -> [B, S/R, H/U, D] -> ring
  attention (Q stays, K/V chunks of the ring group visit) -> inverse
  all-to-all -> [B, S/(U*R), H, D].
* cache-dit "Context Parallelism", USP: Ulysses all-to-all first, ring
  attention on the redistributed data, then the all-to-all reversed.
* edge-dit.cpp "Parallel execution": the decomposition preserves the
  full-attention result exactly.

This composes the oracle's own steps literally; it is checked against plain
``attention.attention`` on the whole sequence.  Values travel as float64
storage (no wire cast), so the only differences from plain attention are
floating-point summation order.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

from . import attention as att
from . import ulysses
from .layout import SPLayout
from .numeric import from_f64, to_f64


def usp_attention(L: SPLayout, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                  scale: Optional[float] = None):
    """q, k, v: float64 [B, S, H, D].  Returns (O [B,S,H,D], per-rank lse).

    The per-rank lse dict maps (r, v) to [B, Hl_v, S_r] (merged over the ring).
    """
    planes = [from_f64(x, "f64") for x in (q, k, v)]
    send = ulysses.s2h_pack(L, planes, "f64", "f64")
    recv = ulysses.a2a(L, "s2h", 3, send)
    ranks = ulysses.s2h_unpack(L, recv, "f64", ("f64", "f64", "f64"))
    o_ranks: Dict[Tuple[int, int], np.ndarray] = {}
    lse_ranks: Dict[Tuple[int, int], np.ndarray] = {}
    for r in range(L.R):
        for vv in range(L.U):
            qr = to_f64(ranks[(r, vv)][0], "f64")
            parts = []
            for j in range(L.R):           # K/V chunks visiting rank (r, vv)
                kj = to_f64(ranks[(j, vv)][1], "f64")
                vj = to_f64(ranks[(j, vv)][2], "f64")
                # sequence-padding rows of the chunk are no keys
                parts.append(att.partial(qr, kj, vj, L.real_rows(j), scale))
            o, lse = att.merge(parts)
            o_ranks[(r, vv)] = from_f64(o, "f64")
            lse_ranks[(r, vv)] = lse
    send_o = ulysses.h2s_pack(L, o_ranks, "f64", "f64")
    recv_o = ulysses.a2a(L, "h2s", 1, send_o)
    out = ulysses.h2s_unpack(L, recv_o, "f64", "f64")
    return to_f64(out, "f64"), lse_ranks
