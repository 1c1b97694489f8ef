"""The Ulysses all-to-all in both directions as an explicit permutation.

Sources:
* edge-dit.cpp "Parallel execution", Ulysses sequence parallelism: Q/K/V
  of shape [B, S/P, H, D] per rank become [B, S, H/P, D] per rank after the
  sequence-to-head all-to-all; the head-to-sequence all-to-all reverses it.
  Packed QKV send path: Q, K and V share one buffer arranged by destination
  rank and destination head group ("peer-major"), optionally converted to a
  16-bit type.  Head-to-sequence path: the output is partitioned by
  destination sequence shard and may be produced directly in BF16/F16.
* SGLang Diffusion "Parallelism Overview", "The Ulysses transport": an
  all-to-all is a permutation, never a reduction, so any transport gives
  bit-identical results.
* cache-dit "Context Parallelism", UAA and "Any Head Num": uneven sequence
  lengths per rank; heads padded to a multiple of U before, unpadded after.

All arrays here hold raw storage bits (uint16 for bf16/f16, uint32 for f32),
so every step that does not convert is bit-exact by construction.  The
layout conventions are those of ``oracle.layout``.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np

from .layout import SPLayout, a2a_counts, buffer_bases
from .numeric import BITS_DTYPE, convert_bits


def _heads_of(L: SPLayout, v: int) -> Tuple[int, int]:
    """Global heads [h0, h1) of head group v that are real (h < H)."""
    h0 = L.head_off[v]
    h1 = min(h0 + L.head_len[v], L.H)
    return h0, max(h0, h1)


def _real(L: SPLayout, off: int, n: int) -> int:
    """How many of the rows [off, off + n) are real (not sequence padding)."""
    return max(0, min(n, L.S - off))


def s2h_pack(L: SPLayout, planes: Sequence[np.ndarray], src_dt: str,
             wire_dt: str) -> np.ndarray:
    """Build every virtual rank's sequence-to-head send buffer.

    planes[p] is the global [B, S, H, D] tensor of plane p (Q, K, V); rank
    (r, u) owns rows [off, off + len) of the S_pad rows.  Its send buffer is,
    for each destination v in order, the block [planes][B][len][Hl_v][D]
    holding head group v of its rows; heads >= H and rows >= S (sequence
    padding) are zero.
    """
    nplanes = len(planes)
    send_base, _, total = buffer_bases(L, "s2h", nplanes)
    send = np.zeros(total, dtype=BITS_DTYPE[wire_dt])
    for r in range(L.R):
        for u in range(L.U):
            rid = L.rank(r, u)
            n, off = L.rank_len[rid], L.rank_off[rid]
            sc, sd, _, _ = a2a_counts(L, "s2h", nplanes, rid)
            m = _real(L, off, n)
            for v in range(L.U):
                blk = np.zeros((nplanes, L.B, n, L.head_len[v], L.D),
                               dtype=BITS_DTYPE[wire_dt])
                h0, h1 = _heads_of(L, v)
                for p in range(nplanes):
                    src = planes[p][:, off:off + m, h0:h1, :]
                    blk[p, :, 0:m, 0:h1 - h0, :] = convert_bits(src, src_dt, wire_dt)
                assert blk.size == sc[v]
                start = send_base[rid] + sd[v]
                send[start:start + blk.size] = blk.reshape(-1)
    return send


def a2a(L: SPLayout, direction: str, nplanes: int, send: np.ndarray) -> np.ndarray:
    """alltoallv inside every Ulysses group: recv[v][from u] = send[u][to v]."""
    send_base, recv_base, total = buffer_bases(L, direction, nplanes)
    recv = np.empty(total, dtype=send.dtype)
    for r in range(L.R):
        for u in range(L.U):            # source
            src = L.rank(r, u)
            sc, sd, _, _ = a2a_counts(L, direction, nplanes, src)
            for v in range(L.U):        # destination
                dst = L.rank(r, v)
                _, _, rc, rd = a2a_counts(L, direction, nplanes, dst)
                assert rc[u] == sc[v]
                a = send_base[src] + sd[v]
                b = recv_base[dst] + rd[u]
                recv[b:b + sc[v]] = send[a:a + sc[v]]
    return recv


def s2h_unpack(L: SPLayout, recv: np.ndarray, wire_dt: str,
               dst_dts: Sequence[str]) -> Dict[Tuple[int, int], List[np.ndarray]]:
    """Head-sharded per-rank planes from the received blocks.

    Returns {(r, v): [plane_0, ...]} with plane_p of shape [B, S_r, Hl_v, D]
    (ring block r's rows in global order, padding rows included, local heads
    of group v), each converted to dst_dts[p].
    """
    nplanes = len(dst_dts)
    _, recv_base, _ = buffer_bases(L, "s2h", nplanes)
    out: Dict[Tuple[int, int], List[np.ndarray]] = {}
    for r in range(L.R):
        Sr = L.ring_len[r]
        for v in range(L.U):
            dst = L.rank(r, v)
            _, _, rc, rd = a2a_counts(L, "s2h", nplanes, dst)
            planes = [np.zeros((L.B, Sr, L.head_len[v], L.D), dtype=BITS_DTYPE[dt])
                      for dt in dst_dts]
            for u in range(L.U):
                n = L.rank_len[L.rank(r, u)]
                row0 = L.rank_off[L.rank(r, u)] - L.ring_off[r]
                a = recv_base[dst] + rd[u]
                blk = recv[a:a + rc[u]].reshape(nplanes, L.B, n, L.head_len[v], L.D)
                for p in range(nplanes):
                    planes[p][:, row0:row0 + n] = convert_bits(blk[p], wire_dt,
                                                               dst_dts[p])
            out[(r, v)] = planes
    return out


def h2s_pack(L: SPLayout, o_ranks: Dict[Tuple[int, int], np.ndarray], src_dt: str,
             wire_dt: str) -> np.ndarray:
    """Head-to-sequence send buffers from each rank's [B, S_r, Hl_v, D] output.

    Rank (r, v) sends peer u the rows of u's slice, all Hl_v local heads;
    local heads whose global index is >= H and sequence-padding rows are
    zero on the wire.
    """
    send_base, _, total = buffer_bases(L, "h2s", 1)
    send = np.zeros(total, dtype=BITS_DTYPE[wire_dt])
    for r in range(L.R):
        for v in range(L.U):
            src = L.rank(r, v)
            sc, sd, _, _ = a2a_counts(L, "h2s", 1, src)
            o = o_ranks[(r, v)]
            h0, h1 = _heads_of(L, v)
            for u in range(L.U):
                n = L.rank_len[L.rank(r, u)]
                m = _real(L, L.rank_off[L.rank(r, u)], n)
                row0 = L.rank_off[L.rank(r, u)] - L.ring_off[r]
                blk = np.zeros((1, L.B, n, L.head_len[v], L.D), dtype=BITS_DTYPE[wire_dt])
                blk[0, :, 0:m, 0:h1 - h0, :] = convert_bits(
                    o[:, row0:row0 + m, 0:h1 - h0, :], src_dt, wire_dt)
                assert blk.size == sc[u]
                start = send_base[src] + sd[u]
                send[start:start + blk.size] = blk.reshape(-1)
    return send


def h2s_unpack(L: SPLayout, recv: np.ndarray, wire_dt: str, out_dt: str) -> np.ndarray:
    """Sequence-sharded output [B, S, H, D]: rank (r, u) fills its real rows
    from every head group v, dropping the padded heads and padding rows."""
    _, recv_base, _ = buffer_bases(L, "h2s", 1)
    out = np.zeros((L.B, L.S, L.H, L.D), dtype=BITS_DTYPE[out_dt])
    for r in range(L.R):
        for u in range(L.U):
            dst = L.rank(r, u)
            n, off = L.rank_len[dst], L.rank_off[dst]
            m = _real(L, off, n)
            _, _, rc, rd = a2a_counts(L, "h2s", 1, dst)
            for v in range(L.U):
                a = recv_base[dst] + rd[v]
                blk = recv[a:a + rc[v]].reshape(1, L.B, n, L.head_len[v], L.D)
                h0, h1 = _heads_of(L, v)
                out[:, off:off + m, h0:h1, :] = convert_bits(
                    blk[0, :, 0:m, 0:h1 - h0, :], wire_dt, out_dt)
    return out
