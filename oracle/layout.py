"""Sequence split, head padding and all-to-all bookkeeping (integers only).

Sources:
* edge-dit.cpp "Parallel execution", SPSequenceSplit: each rank owns a local
  slice of the sequence, recorded with its length and offset; and
  SPAllToAll4DLayout: the per-peer element counts of each redistribution.
* cache-dit "Context Parallelism", UAA: sequence lengths that do not divide
  by the Ulysses degree are allowed, so ranks hold different lengths; and
  "Any Head Num": the head count is padded up to a multiple of the degree
  before the all-to-all and unpadded after it.
* SGLang Diffusion "Parallelism Overview", "What happens to the shapes": the
  sequence is split outer by ring degree R and inner by Ulysses degree U;
  ranks of one Ulysses group are contiguous, ring groups are strided.

Readings where the pages are silent:
* The uneven split is the balanced one: of n parts, the first S mod n get
  one extra row.
* Padded heads are appended after the real heads (global heads H..Hp-1).
* Virtual rank id = r*U + u, so that ids in order partition the sequence in
  order (ring blocks outer, Ulysses ranks inner).
* Wire blocks are peer-major and plane-major inside: the block that rank u
  of ring group r sends to rank v is [planes][B][L_(r,u)][Hl_v][D].

Two alternate layouts of the same permutation:
* cache-dit "Context Parallelism", the padding-free variant of "Any Head
  Num": the heads are not padded; rank v gets Hl_v heads of a balanced split
  of H (the first H mod U ranks one more), and the all-to-all counts follow.
  (cache-dit allows it only when the sequence divides evenly; the exact
  counts here need no such condition.)
* xLLM "DiT Architecture and Capability Matrix": with sequence parallelism
  the total sequence length is padded to a multiple of lcm(SP, 64) before
  partitioning.  Reading: SP = U * R, the padding rows are appended after the
  real rows, split evenly with them, travel as zeros, are excluded from
  attention and are dropped from the output.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Tuple


def balanced_split(S: int, n: int) -> Tuple[List[int], List[int]]:
    """Lengths and offsets of S rows over n ranks, first S%n ranks get +1."""
    if n < 1 or S < 0:
        raise ValueError("need n >= 1 and S >= 0")
    base, extra = divmod(S, n)
    lens = [base + (1 if i < extra else 0) for i in range(n)]
    offs = []
    acc = 0
    for L in lens:
        offs.append(acc)
        acc += L
    return lens, offs


def lcm(a: int, b: int) -> int:
    from math import gcd
    return a * b // gcd(a, b)


def padded_length(S: int, sp: int) -> int:
    """S rounded up to a multiple of lcm(sp, 64)."""
    m = lcm(sp, 64)
    return -(-S // m) * m


def padded_heads(H: int, U: int) -> Tuple[int, int]:
    """(Hp, Hl): H rounded up to a multiple of U, and heads per rank."""
    Hl = -(-H // U)
    return Hl * U, Hl


@dataclass(frozen=True)
class SPLayout:
    B: int
    S: int                          # real rows of the sequence
    H: int
    D: int
    U: int
    R: int
    Hp: int                         # head slots on the wire and in the head layout
    Hl: int                         # the largest head group
    ring_len: Tuple[int, ...]       # [R], over the S_pad rows
    ring_off: Tuple[int, ...]
    rank_len: Tuple[int, ...]       # [R*U], id = r*U + u
    rank_off: Tuple[int, ...]       # global row offset of the rank's slice
    head_len: Tuple[int, ...]       # [U] heads of group v
    head_off: Tuple[int, ...]       # first head slot of group v
    S_pad: int                      # rows split over the ranks (>= S)
    pad_heads: bool = True
    pad_lcm64: bool = False

    def rank(self, r: int, u: int) -> int:
        return r * self.U + u

    def heads(self, v: int) -> slice:
        return slice(self.head_off[v], self.head_off[v] + self.head_len[v])

    def real_rows(self, r: int) -> int:
        """Rows of ring block r that are not sequence padding."""
        return max(0, min(self.S - self.ring_off[r], self.ring_len[r]))

    @property
    def S_cap(self) -> int:
        return max(self.ring_len) if self.ring_len else 0


def make_layout(B: int, S: int, H: int, D: int, U: int, R: int,
                pad_heads: bool = True, pad_lcm64: bool = False) -> SPLayout:
    """pad_heads: heads padded to a multiple of U (else a balanced split of
    the H real heads); pad_lcm64: the sequence padded to a multiple of
    lcm(U*R, 64) before the split."""
    if min(B, H, D, U, R) < 1 or S < 0:
        raise ValueError("bad sizes")
    S_pad = padded_length(S, U * R) if pad_lcm64 else S
    ring_len, ring_off = balanced_split(S_pad, R)
    rank_len: List[int] = []
    rank_off: List[int] = []
    for r in range(R):
        lens, offs = balanced_split(ring_len[r], U)
        rank_len.extend(lens)
        rank_off.extend(ring_off[r] + o for o in offs)
    if pad_heads:
        Hp, Hl = padded_heads(H, U)
        head_len, head_off = [Hl] * U, [v * Hl for v in range(U)]
    else:
        head_len, head_off = balanced_split(H, U)
        Hp, Hl = H, max(head_len)
    return SPLayout(B, S, H, D, U, R, Hp, Hl, tuple(ring_len), tuple(ring_off),
                    tuple(rank_len), tuple(rank_off), tuple(head_len), tuple(head_off), S_pad,
                    pad_heads, pad_lcm64)


def a2a_counts(L: SPLayout, direction: str, nplanes: int, rank_id: int):
    """alltoallv argument set of one virtual rank, in elements.

    Returns (send_counts, send_displs, recv_counts, recv_displs), each of
    length U, indexed by the peer's Ulysses index inside the rank's ring
    group.  direction is "s2h" (sequence-sharded -> head-sharded) or "h2s".
    """
    U = L.U
    r, me = divmod(rank_id, U)

    def per_row(v):                  # elements of one row of head group v
        return nplanes * L.B * L.head_len[v] * L.D

    def rows(u):
        return L.rank_len[r * U + u]

    if direction == "s2h":
        # I send rows(me) rows of every peer's head group; I receive, from
        # each peer u, rows(u) rows of my head group.
        sc = [per_row(v) * rows(me) for v in range(U)]
        rc = [per_row(me) * rows(u) for u in range(U)]
    elif direction == "h2s":
        # I send each peer u its rows(u) rows of my head group; I receive
        # rows(me) rows of each peer's head group.
        sc = [per_row(me) * rows(u) for u in range(U)]
        rc = [per_row(v) * rows(me) for v in range(U)]
    else:
        raise ValueError(direction)
    sd, rd = [], []
    acc = 0
    for c in sc:
        sd.append(acc)
        acc += c
    acc = 0
    for c in rc:
        rd.append(acc)
        acc += c
    return sc, sd, rc, rd


def buffer_bases(L: SPLayout, direction: str, nplanes: int):
    """Element offset of each virtual rank's send and recv buffer when all
    ranks' buffers are laid end to end in id order (one HBM allocation)."""
    n = L.R * L.U
    send_base, recv_base = [], []
    s_acc = r_acc = 0
    for rid in range(n):
        sc, _, rc, _ = a2a_counts(L, direction, nplanes, rid)
        send_base.append(s_acc)
        recv_base.append(r_acc)
        s_acc += sum(sc)
        r_acc += sum(rc)
    return send_base, recv_base, s_acc
