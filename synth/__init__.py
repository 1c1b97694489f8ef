"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only draws random numbers and names workload shapes.  It holds
none of the method's arithmetic (no attention, no layout permutation, no
guidance combine), so that the oracle and the CUDA path can both consume the
same inputs without sharing any of the computation they are compared on.

Values are drawn with numpy's PCG64 generator (``numpy.random.default_rng``)
as float32 standard normals, multiplied by the workload's scale, and then
converted to the workload's storage type by PyTorch's CPU conversion
(round-to-nearest-even).  The returned tensors live in host memory; callers
move them to the device themselves.

The workloads stand in for the pages' FLUX.1-dev, Qwen-Image and Wan2.1
pipelines (cache-dit "Context Parallelism" and diffusers "Distributed
inference" benchmark tables): no weights, prompts or datasets are involved,
only tensors of the shapes those models feed to attention.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np
import torch

_TORCH_DTYPES = {
    "f32": torch.float32,
    "bf16": torch.bfloat16,
    "f16": torch.float16,
}

# Seed offsets for the five tensors a workload draws.  Every workload's base
# seed is 0; Q, K, V, the unconditional and the conditional branch use
# base+0 .. base+4.
SEED_Q, SEED_K, SEED_V, SEED_UNCOND, SEED_COND = range(5)


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


def normal(shape: Tuple[int, ...], seed: int, scale: float = 1.0,
           dtype: str = "f32") -> torch.Tensor:
    """Host tensor of N(0,1)*scale values in ``dtype``, drawn from ``seed``."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    t = torch.from_numpy(x)
    if dtype != "f32":
        t = t.to(_TORCH_DTYPES[dtype])
    return t


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a host tensor (every f32/bf16/f16 value is a double)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def as_bits(t: torch.Tensor) -> np.ndarray:
    """Raw storage bits of a host tensor as an unsigned numpy array."""
    t = t.detach().to("cpu").contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.element_size() == 4:
        return t.view(torch.int32).numpy().view(np.uint32)
    raise ValueError("unsupported element size")


def digest(*tensors: torch.Tensor) -> str:
    """First 16 hex digits of the SHA-256 of the tensors' raw bytes, in
    order: a record of exactly which inputs a run used."""
    import hashlib
    h = hashlib.sha256()
    for t in tensors:
        h.update(as_bits(t).tobytes())
    return h.hexdigest()[:16]


def _tables(angles: np.ndarray):
    """float32 cos/sin tables of float64 angles [S, D/2] (RNE to float32)."""
    return (torch.from_numpy(np.cos(angles).astype(np.float32)),
            torch.from_numpy(np.sin(angles).astype(np.float32)))


def rope_tables_linear(S: int, D: int, base: float = 10000.0):
    """Rotary angle tables of a 1-D position index: token t, pair i has the
    angle t * base**(-2i/D).  Every token has distinct angles, which makes it
    the stronger test input."""
    i = np.arange(D // 2, dtype=np.float64)
    t = np.arange(S, dtype=np.float64)[:, None]
    return _tables(t * base ** (-2.0 * i / D))


def rope_axes(D: int) -> Tuple[int, int, int]:
    """Head-dim split of the three-axis position ids (16, 56, 56 for D=128)."""
    a0 = 2 * max(1, D // 16)
    a1 = 2 * ((D - a0) // 4)
    return a0, a1, D - a0 - a1


def rope_tables_joint(S_txt: int, S: int, D: int, base: float = 10000.0):
    """Rotary angle tables of a joint text+image sequence with three-axis
    position ids, the stand-in for the FLUX-family models' positions: text
    tokens have ids (0, 0, 0), image token k of a w-wide grid (0, k // w,
    k % w), w = ceil(sqrt(S - S_txt)).  Axis a owns rope_axes(D)[a] of the
    head dims; its pair j turns by id_a * base**(-2j/d_a)."""
    n = S - S_txt
    w = max(1, int(np.ceil(np.sqrt(n)))) if n > 0 else 1
    k = np.arange(n)
    ids = np.zeros((S, 3), dtype=np.float64)
    ids[S_txt:, 1] = k // w
    ids[S_txt:, 2] = k % w
    cols = []
    for a, da in enumerate(rope_axes(D)):
        j = np.arange(da // 2, dtype=np.float64)
        cols.append(ids[:, a:a + 1] * base ** (-2.0 * j / da))
    return _tables(np.concatenate(cols, axis=1))


@dataclass(frozen=True)
class Workload:
    """One attention workload: shapes, parallel degrees and value recipe."""

    name: str
    B: int
    S: int
    H: int
    D: int
    dtype: str                      # storage type of Q/K/V
    scale: float                    # N(0,1) multiplier for Q/K/V
    U: Tuple[int, ...]              # Ulysses degrees exercised
    R: int                          # ring degree
    cfg_shape: Tuple[int, ...]      # [2, ...]: uncond, cond
    cfg_in: str
    cfg_out: str
    g: float
    seed: int = 0
    note: str = ""
    S_txt: int = 0                  # text tokens at the head of the joint sequence

    def qkv(self, device: Optional[str] = None):
        shp = (self.B, self.S, self.H, self.D)
        out = tuple(normal(shp, self.seed + s, self.scale, self.dtype)
                    for s in (SEED_Q, SEED_K, SEED_V))
        if device is not None:
            out = tuple(t.to(device) for t in out)
        return out

    def cfg_pair(self):
        """Stacked [2, ...] host tensor: index 0 unconditional, 1 conditional."""
        one = self.cfg_shape[1:]
        u = normal(one, self.seed + SEED_UNCOND, 1.0, self.cfg_in)
        c = normal(one, self.seed + SEED_COND, 1.0, self.cfg_in)
        return torch.stack([u, c])

    @property
    def attn_flops(self) -> float:
        """Algorithmic attention work: 4*B*H*S^2*D (real heads and rows only)."""
        return 4.0 * self.B * self.H * float(self.S) ** 2 * self.D


WORKLOADS = {
    "tiny": Workload("tiny", 1, 256, 4, 64, "f32", 1.0, (2,), 2,
                     (2, 1, 256, 4, 64), "f32", "f32", 4.0,
                     note="fp32 path, U=2 and R=2, also USP 2x2"),
    "flux1024": Workload("flux1024", 1, 4608, 24, 128, "bf16", 0.5, (2, 4), 1,
                         (2, 4608, 3072), "bf16", "bf16", 3.5,
                         note="4096 image + 512 text tokens", S_txt=512),
    "flux1008": Workload("flux1008", 1, 4481, 24, 128, "bf16", 0.5, (4,), 2,
                         (2, 4481, 3072), "bf16", "bf16", 3.5,
                         note="63x63=3969 image + 512 text tokens; uneven", S_txt=512),
    "flux1008_4480": Workload("flux1008_4480", 1, 4480, 24, 128, "bf16", 0.5,
                              (4,), 2, (2, 4480, 3072), "bf16", "bf16", 3.5,
                              note="the literal 3969 + 511 token count", S_txt=511),
    "qwen1328": Workload("qwen1328", 2, 7145, 24, 128, "bf16", 0.5, (5,), 2,
                         (2, 7145, 3072), "f32", "bf16", 4.0,
                         note="83x83=6889 image + 256 text tokens; 24 heads "
                              "padded to 25 for U=5", S_txt=256),
    "wan": Workload("wan", 1, 75600, 40, 128, "bf16", 0.5, (8,), 4,
                    (2, 75600, 5120), "bf16", "bf16", 5.0,
                    note="21 latent frames x 45x80 tokens; U=8 x R=4"),
}
