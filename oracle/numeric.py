"""Round-to-nearest-even conversions used by the casts the method allows.

The pages let the packed all-to-all path convert F32 to a 16-bit wire type
and let the head-to-sequence path emit BF16/F16 output directly (edge-dit.cpp
"Parallel execution", packed QKV send path and head-to-sequence path).  They
do not name a rounding mode; IEEE-754 round-to-nearest-even is the plain
reading and is what this oracle implements.

``f64_to_bf16_bits`` rounds a double straight to bfloat16 (no intermediate
float32) by scaling it to the bfloat16 grid at its binade, which is exact.
``f64_to_f16_bits`` uses numpy's correctly rounded double->half conversion.
"""
from __future__ import annotations

import numpy as np

_BF16_MANT = 7          # stored mantissa bits of bfloat16


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (the upper half of a float32)."""
    b32 = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16))
    return b32.view(np.float32).astype(np.float64)


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def f32_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint32).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (nearest, ties to even); return bits.

    Works on the sign/exponent/mantissa fields of binary64:
      * NaN stays a (quiet) NaN, +-inf stays +-inf;
      * values whose rounded magnitude reaches 2^128 overflow to inf;
      * values below the smallest bfloat16 normal round into the subnormal
        grid (spacing 2^-133), which is how a float32 holds them too.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat = x.reshape(-1)
    o = out.reshape(-1)
    u = flat.view(np.uint64)
    sign = ((u >> np.uint64(63)) & np.uint64(1)).astype(np.uint16) << np.uint16(15)
    nan = np.isnan(flat)
    inf = np.isinf(flat)
    a = np.abs(flat)
    res = np.zeros(flat.shape, dtype=np.uint16)
    fin = ~(nan | inf)
    # Exact rounding on the real line: the bfloat16 grid spacing at |x| is
    # 2^(e-7) for normal x with exponent e, and 2^-133 below 2^-126.
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        _, e2 = np.frexp(a)                      # a = f * 2^e2, f in [0.5, 1)
        e = e2.astype(np.int64) - 1              # a in [2^e, 2^(e+1))
        e = np.maximum(e, -126)                  # subnormal range shares 2^-133
        ulp_exp = e - _BF16_MANT
        q = np.ldexp(a, -ulp_exp)                # a / ulp, exact (power of 2)
        qf = np.floor(q)
        frac = q - qf
        up = (frac > 0.5) | ((frac == 0.5) & (np.mod(qf, 2.0) == 1.0))
        qr = qf + up.astype(np.float64)
        r = np.ldexp(qr, ulp_exp)                # rounded magnitude, exact
    over = fin & (r >= 2.0 ** 128)
    ok = fin & ~over
    # Re-encode the rounded magnitude (exactly a bfloat16 value) through
    # float32, which holds every bfloat16 value exactly.
    r32 = r[ok].astype(np.float32).view(np.uint32)
    res[ok] = (r32 >> np.uint32(16)).astype(np.uint16)
    res[over | inf] = np.uint16(0x7F80)
    res[nan] = np.uint16(0x7FC0)
    o[:] = res | np.where(nan, np.uint16(0), sign)
    return out


def f64_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to IEEE binary16 (nearest even) via numpy; return bits."""
    with np.errstate(over="ignore", invalid="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def f64_to_f32_bits(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore", invalid="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)


BITS_DTYPE = {"f64": np.uint64, "f32": np.uint32, "bf16": np.uint16,
              "f16": np.uint16}


def to_f64(bits: np.ndarray, dt: str) -> np.ndarray:
    if dt == "f64":
        return np.asarray(bits, dtype=np.uint64).view(np.float64).copy()
    if dt == "f32":
        return f32_bits_to_f64(bits)
    if dt == "bf16":
        return bf16_bits_to_f64(bits)
    if dt == "f16":
        return f16_bits_to_f64(bits)
    raise ValueError(dt)


def from_f64(x: np.ndarray, dt: str) -> np.ndarray:
    if dt == "f64":
        return np.asarray(x, dtype=np.float64).copy().view(np.uint64)
    if dt == "f32":
        return f64_to_f32_bits(x)
    if dt == "bf16":
        return f64_to_bf16_bits(x)
    if dt == "f16":
        return f64_to_f16_bits(x)
    raise ValueError(dt)


def convert_bits(bits: np.ndarray, src: str, dst: str) -> np.ndarray:
    """Storage conversion src->dst: exact when widening, RNE when narrowing.

    Identity conversions return the input bits untouched, so a pure
    permutation stays bit-exact even for NaN payloads.
    """
    if src == dst:
        return np.asarray(bits, dtype=BITS_DTYPE[dst]).copy()
    return from_f64(to_f64(bits, src), dst)
