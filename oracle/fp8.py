"""FP8 (e4m3) wire format for the Ulysses all-to-all.

Source: cache-dit "Context Parallelism", Async FP8 Ulysses Attention: the
all-to-all of Q, V and the attention output O travels in float8, while K stays
in FP16/BF16 because the softmax of Q K^T is sensitive to its precision.  The
pages give neither the float8 variant nor the scaling.  Reading: e4m3 (4
exponent bits, bias 7, 3 mantissa bits, no infinities, largest finite 448, one
NaN code per sign), one scale per (token, head): s = amax / 448 over the head's
D values, codes = e4m3(x * (1/s)), value = code * s.  Every step that decides a
code is done in float32, as the kernel does (numpy float32 arithmetic is IEEE
round-to-nearest-even, like the GPU's): amax, s = fl32(amax / 448),
r = fl32(1 / s), y = fl32(x * r), code = round-to-nearest-even e4m3 of y with
saturation to +-448.  Decoding: fl32(value(code) * s).  A head whose amax is
zero has s = 0 and zero codes.

The wire record of one (token, head): D code bytes, then s as a float32,
then 12 zero bytes (16-byte aligned records).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_value(code: np.ndarray) -> np.ndarray:
    """float64 value of e4m3 codes (uint8) from the format's definition."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = sign * np.exp2(e - 7.0) * (1.0 + m / 8.0)
    sub = sign * np.exp2(-6.0) * (m / 8.0)
    v = np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


_POS_CODES = np.arange(0x7F, dtype=np.uint8)           # every finite non-negative code
_POS_VALUES = e4m3_value(_POS_CODES)                     # increasing


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even to e4m3 with saturation to +-448 (finite values
    beyond 448 give 448); NaN gives the NaN code."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    idx = np.searchsorted(_POS_VALUES, np.minimum(a, E4M3_MAX), side="left")
    idx = np.clip(idx, 0, len(_POS_VALUES) - 1)
    hi = idx                                             # first value >= a
    lo = np.maximum(idx - 1, 0)
    d_lo = np.abs(a - _POS_VALUES[lo])
    d_hi = np.abs(_POS_VALUES[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(np.signbit(y), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(y), np.uint8(0x7F), code).astype(np.uint8)


def quantize_heads(x: np.ndarray):
    """Per-head quantization of float32 values x [..., D]: (codes uint8
    [..., D], scales float32 [...])."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    with np.errstate(divide="ignore"):
        r = np.where(s > 0, np.float32(1.0) / s, np.float32(0.0)).astype(np.float32)
    y = (x * r[..., None]).astype(np.float32)
    return e4m3_encode(y), s


def dequantize_heads(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    """float32 values code * s of [..., D] codes and [...] scales."""
    v = e4m3_value(codes).astype(np.float32)            # every e4m3 value is a float32
    return (v * np.asarray(s, dtype=np.float32)[..., None]).astype(np.float32)


def record_bytes(D: int) -> int:
    return D + 16


def to_records(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Wire records [..., D + 16] (uint8) of codes [..., D] and scales [...]."""
    D = codes.shape[-1]
    rec = np.zeros(codes.shape[:-1] + (record_bytes(D),), dtype=np.uint8)
    rec[..., :D] = codes
    rec[..., D:D + 4] = np.asarray(s, dtype=np.float32)[..., None].view(np.uint8)
    return rec


def from_records(rec: np.ndarray):
    """(codes [..., D], scales [...]) of wire records [..., D + 16]."""
    D = rec.shape[-1] - 16
    codes = rec[..., :D]
    s = np.ascontiguousarray(rec[..., D:D + 4]).view(np.float32)[..., 0]
    return codes, s


# ---- the all-to-all with an FP8 wire --------------------------------------
# A record is D + 16 bytes; seen as (D + 16) / 2 16-bit words, the records of
# one (plane, batch, row) form exactly the run of a 16-bit wire whose head dim
# is (D + 16) / 2, so the permutation is ``oracle.ulysses``'s, on words.

def _word_layout(L):
    from .layout import make_layout
    return make_layout(L.B, L.S, L.H, record_bytes(L.D) // 2, L.U, L.R, pad_heads=L.pad_heads,
                       pad_lcm64=L.pad_lcm64)


def _words(rec: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(rec).view(np.uint16)


def _recs(words: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(words).view(np.uint8)


def s2h_pack(L, planes, src_dt: str) -> np.ndarray:
    """Send buffers (uint16 words) of the seq->head exchange: every head of
    every plane ([B, S, H, D] storage bits of src_dt) quantized to a record."""
    from . import numeric, ulysses
    words = []
    for bits in planes:
        x = numeric.to_f64(bits, src_dt).astype(np.float32)
        codes, s = quantize_heads(x)
        words.append(_words(to_records(codes, s)))
    return ulysses.s2h_pack(_word_layout(L), words, "bf16", "bf16")


def a2a(L, direction: str, nplanes: int, send: np.ndarray) -> np.ndarray:
    from . import ulysses
    return ulysses.a2a(_word_layout(L), direction, nplanes, send)


def s2h_unpack(L, recv: np.ndarray, dst_dts):
    """{(r, v): [plane bits in dst_dts[p], shape [B, S_r, Hl, D]]}: the
    received records decoded."""
    from . import numeric, ulysses
    n = len(dst_dts)
    ranks = ulysses.s2h_unpack(_word_layout(L), recv, "bf16", ["bf16"] * n)
    out = {}
    for key, planes in ranks.items():
        res = []
        for p, dt in enumerate(dst_dts):
            codes, s = from_records(_recs(planes[p]))
            res.append(numeric.from_f64(dequantize_heads(codes, s).astype(np.float64), dt))
        out[key] = res
    return out


def h2s_pack(L, o_ranks, src_dt: str) -> np.ndarray:
    """Send buffers of the head->seq exchange from each rank's [B, S_r, Hl, D]
    output bits (src_dt); padded heads travel as zero records."""
    from . import numeric, ulysses
    words = {}
    for key, bits in o_ranks.items():
        x = numeric.to_f64(bits, src_dt).astype(np.float32)
        codes, s = quantize_heads(x)
        words[key] = _words(to_records(codes, s))
    return ulysses.h2s_pack(_word_layout(L), words, "bf16", "bf16")


def h2s_unpack(L, recv: np.ndarray, out_dt: str) -> np.ndarray:
    """Sequence-layout output [B, S, H, D] (bits of out_dt) from the received
    records, padded heads dropped."""
    from . import numeric, ulysses
    words = ulysses.h2s_unpack(_word_layout(L), recv, "bf16", "bf16")
    codes, s = from_records(_recs(words))
    return numeric.from_f64(dequantize_heads(codes, s).astype(np.float64), out_dt)
