"""Exact attention, the partial over one key chunk, and the log-sum-exp merge.

Sources:
* edge-dit.cpp "Parallel execution", Ulysses sequence parallelism: each rank
  computes O = softmax(Q K^T / sqrt(D)) V over the full sequence for its
  heads; the result is exact, not an approximation.  No mask appears and
  DiT attention is bidirectional.
* SGLang Diffusion "Parallelism Overview", "What happens to the shapes" and
  "Constraints": ring attention keeps Q in place while K/V chunks visit, and
  the per-hop merge needs each kernel call's softmax log-sum-exp; ranks of a
  ring group hold the same heads over different rows, so the merge is an
  online-softmax combination.  The masked text path and replicated prefix
  are attended once and folded in "with the same online-softmax merge".
* diffusers "Distributed inference", Ring Anything Attention: K/V padded to
  a common length are trimmed to each rank's real length before attention;
  attention masks are not supported (attn_mask must be None).

Readings (the pages give no formula beyond the softmax line):
* scale defaults to 1/sqrt(D).
* log-sum-exp is natural-log: lse_i = ln sum_j exp(s_ij).
* A partial's O is normalised by its own chunk's softmax denominator; the
  merge rescales it by exp(lse_chunk - lse_total).  Keys past the chunk's
  valid length are excluded, never zero-filled into the sum.
* An empty chunk has lse = -inf and O = 0, and drops out of a merge.

Arrays are float64 numpy; q is [B, Sq, H, D], k and v are [B, Sk, H, D].
"""
from __future__ import annotations

import math
from typing import Optional, Sequence, Tuple

import numpy as np


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
              scale: Optional[float] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Exact softmax attention: returns (O [B,Sq,H,D], lse [B,H,Sq])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = np.zeros((B, Sq, H, v.shape[3]), dtype=np.float64)
    lse = np.full((B, H, Sq), -np.inf, dtype=np.float64)
    if Sk == 0:
        return o, lse
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, :, h, :] @ k[b, :, h, :].T)        # [Sq, Sk]
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            den = e.sum(axis=1, keepdims=True)
            o[b, :, h, :] = (e @ v[b, :, h, :]) / den
            lse[b, h, :] = m[:, 0] + np.log(den[:, 0])
    return o, lse


def partial(q: np.ndarray, k_chunk: np.ndarray, v_chunk: np.ndarray,
            sk_valid: Optional[int] = None,
            scale: Optional[float] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Attention of q against the first sk_valid keys of one K/V chunk.

    O is normalised by the chunk's own denominator; lse is the chunk's
    log-sum-exp.  Rows of the chunk at or past sk_valid (padding) are
    excluded from the softmax entirely.
    """
    if sk_valid is None:
        sk_valid = k_chunk.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[3])
    return attention(q, k_chunk[:, :sk_valid], v_chunk[:, :sk_valid], scale)


def merge(parts: Sequence[Tuple[np.ndarray, np.ndarray]]) -> Tuple[np.ndarray, np.ndarray]:
    """Fold partials (O_r [B,Sq,H,D], lse_r [B,H,Sq]) into the exact result.

    lse = M + ln sum_r exp(lse_r - M) with M = max_r lse_r, and
    O = sum_r exp(lse_r - lse) * O_r, accumulated for r ascending.
    Rows whose every part is empty (all lse_r = -inf) give O = 0, lse = -inf.
    """
    if not parts:
        raise ValueError("merge needs at least one partial")
    o0, l0 = parts[0]
    lses = np.stack([np.asarray(l, dtype=np.float64) for _, l in parts])  # [R,B,H,Sq]
    M = lses.max(axis=0)
    empty = np.isneginf(M)
    Msafe = np.where(empty, 0.0, M)
    with np.errstate(invalid="ignore"):
        w = np.exp(lses - Msafe[None])                 # exp(-inf) = 0
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, Msafe + np.log(np.where(empty, 1.0, tot)))
    o = np.zeros(np.shape(o0), dtype=np.float64)
    for r, (o_r, _) in enumerate(parts):
        with np.errstate(invalid="ignore"):
            wr = np.where(empty, 0.0, np.exp(lses[r] - np.where(empty, 0.0, lse)))
        # weights are per (b, h, i); O is laid out [b, i, h, d]
        o += np.transpose(wr, (0, 2, 1))[..., None] * np.asarray(o_r, dtype=np.float64)
    return o, lse


def masked(q: np.ndarray, k: np.ndarray, v: np.ndarray, key_mask: np.ndarray,
           scale: Optional[float] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Attention where query rows see only the keys their mask allows.

    key_mask: bool [B, Sq, Sk] (True = the key takes part) or [B, Sk] (the
    same keys for every query).  Source: SGLang Diffusion "Parallelism
    Overview", Constraints: the masked / tail-padded text path (text tokens
    padded to a fixed length, the padding excluded as keys); xLLM "DiT
    Architecture and Capability Matrix": packed data with live/padding
    boundaries, padding excluded.  A row with no allowed key gives O = 0 and
    lse = -inf, as an empty chunk does.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, H, D = q.shape
    mask = np.asarray(key_mask, dtype=bool)
    if mask.ndim == 2:
        mask = np.broadcast_to(mask[:, None, :], (B, Sq, mask.shape[1]))
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = np.zeros((B, Sq, H, v.shape[3]), dtype=np.float64)
    lse = np.full((B, H, Sq), -np.inf, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, :, h, :] @ k[b, :, h, :].T)
            s = np.where(mask[b], s, -np.inf)
            m = s.max(axis=1, keepdims=True) if s.shape[1] else np.full((Sq, 1), -np.inf)
            live = np.isfinite(m[:, 0])
            msafe = np.where(np.isfinite(m), m, 0.0)
            e = np.exp(s - msafe)                        # exp(-inf) = 0 for masked keys
            den = e.sum(axis=1, keepdims=True)
            with np.errstate(invalid="ignore", divide="ignore"):
                o[b, :, h, :] = np.where(live[:, None], (e @ v[b, :, h, :]) / den, 0.0)
                lse[b, h, :] = np.where(live, msafe[:, 0] + np.log(den[:, 0]), -np.inf)
    return o, lse


def varlen(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_q: Sequence[int], cu_k: Sequence[int],
           scale: Optional[float] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Attention of packed variable-length sequences: q [Tq, H, D], k and v
    [Tk, H, D]; sequence s has queries [cu_q[s], cu_q[s+1]) and keys
    [cu_k[s], cu_k[s+1]), and attends only to its own keys.  Returns
    (O [Tq, H, D], lse [H, Tq]).  Source: SGLang Diffusion "Parallelism
    Overview", the generic varlen path (several packed segments per row);
    xLLM, packed TND data with live/padding boundaries.  Query rows outside
    every sequence are not written (O = 0, lse = -inf here).
    """
    q = np.asarray(q, dtype=np.float64)
    Tq, H, D = q.shape
    o = np.zeros((Tq, H, np.shape(v)[2]), dtype=np.float64)
    lse = np.full((H, Tq), -np.inf, dtype=np.float64)
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        if q1 == q0:
            continue
        os_, ls_ = attention(q[None, q0:q1], np.asarray(k)[None, k0:k1], np.asarray(v)[None, k0:k1], scale)
        o[q0:q1] = os_[0]
        lse[:, q0:q1] = ls_[0]
    return o, lse
