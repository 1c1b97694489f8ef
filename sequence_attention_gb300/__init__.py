"""GB300 sequence-parallel DiT attention hot path: Python binding of libditsp.

Each function here has the name of the C entry point it calls and only
marshals arguments: tensor pointers, strides and element types go in, the
CUDA kernels of libditsp.so do all of the work on the caller's current CUDA
stream.  PyTorch is used for device memory and streams only.  There is no
CPU or PyTorch fallback: if the library is missing, importing raises.

Tensor conventions (element strides are read from the tensors, the head dim
must be contiguous):
  Q of the query blocks         [n_q,  B, S, H, D]
  K, V of the key/value blocks  [n_kv, B, S, H, D]
  partial outputs               [n_q, n_kv, B, S, H, D]
  partial log-sum-exp           [n_q, n_kv, B, H, S]   (float32)

Wire buffers are flat tensors; a uint8 wire buffer carries the e4m3 record
format (DIT_E4M3, Layout.wire_bytes_e4m3 bytes), any other dtype its own.
"""
from __future__ import annotations

import ctypes
import math
from ctypes import byref, c_int, c_int64, c_void_p
from typing import List, Optional, Sequence

import torch

from . import _lib
from ._lib import (DIT_BF16, DIT_E4M3, DIT_F16, DIT_F32, DIT_HEAD_TO_SEQ, DIT_SEQ_TO_HEAD, DitError,
                   DitLseView, DitSpLayout, DitView, check, lib)

__all__ = [
    "DitError", "Layout", "DIT_SEQ_TO_HEAD", "DIT_HEAD_TO_SEQ", "DIT_E4M3",
    "dit_sp_layout_init", "dit_sp_a2a_counts", "dit_ulysses_pack", "dit_a2a_sim",
    "dit_ulysses_unpack", "dit_attn_partial", "dit_attn_merge_lse", "dit_attention",
    "dit_cfg_combine", "dit_device_status", "library_path", "dit_sp_signal", "dit_a2a_sim_checked",
    "dit_ulysses_pack_joint", "dit_ulysses_unpack_joint", "dit_ulysses_unpack_rope", "dit_attn_varlen",
    "dit_ulysses_seq_to_head", "dit_ulysses_head_to_seq", "dit_attn_ring", "dit_attn_ring_rows",
    "dit_attn_ring_merge_static",
]

lib()   # load now: fail at import time, not at first call

_DT = {torch.float32: DIT_F32, torch.bfloat16: DIT_BF16, torch.float16: DIT_F16, torch.uint8: DIT_E4M3}


def library_path() -> str:
    return _lib.LIB_PATH


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _stream(stream) -> c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return c_void_p(s.cuda_stream)


def _addr(t: torch.Tensor) -> int:
    """The device address of t: every buffer the kernels touch must live on a
    CUDA device (a host pointer would fault the GPU, so it is refused here)."""
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    return t.data_ptr()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else c_void_p(_addr(t))


class Layout:
    """A filled dit_sp_layout plus the buffer shapes it implies."""

    def __init__(self, raw: DitSpLayout):
        self.raw = raw

    def __getattr__(self, name):
        raw = self.__dict__["raw"]
        v = getattr(raw, name)
        if name in ("ring_len", "ring_off", "ring_real"):
            return list(v)[: raw.R]
        if name in ("rank_len", "rank_off"):
            return list(v)[: raw.R * raw.U]
        if name in ("head_len", "head_off"):
            return list(v)[: raw.U]
        return v

    def real_rows(self, r: int) -> int:
        """Rows of ring block r that are not sequence padding (the layout's
        ring_real, filled by dit_sp_layout_init)."""
        return self.raw.ring_real[r]

    def head_shape(self):
        """Head-layout plane [R, B, S_cap, Hp, D]."""
        r = self.raw
        return (r.R, r.B, r.S_cap, r.Hp, r.D)

    def seq_shape(self):
        r = self.raw
        return (r.B, r.S, r.H, r.D)

    def wire_elems(self, nplanes: int) -> int:
        r = self.raw
        return nplanes * r.B * r.S_pad * r.Hp * r.D

    def wire_bytes_e4m3(self, nplanes: int) -> int:
        """Bytes of an e4m3 wire: one (D + 16)-byte record per (token, head)."""
        r = self.raw
        return nplanes * r.B * r.S_pad * r.Hp * (r.D + 16)


def dit_sp_layout_init(B: int, S: int, H: int, D: int, U: int, R: int, pad_heads: bool = True,
                       pad_lcm64: bool = False) -> Layout:
    """pad_heads=False: the padding-free uneven head split; pad_lcm64: the
    sequence padded to a multiple of lcm(U*R, 64)."""
    raw = DitSpLayout()
    flags = (0 if pad_heads else _lib.DIT_LAYOUT_NOPAD_HEADS) | (_lib.DIT_LAYOUT_PAD_LCM64 if pad_lcm64 else 0)
    check(lib().dit_sp_layout_init_ex(B, S, H, D, U, R, flags, byref(raw)))
    return Layout(raw)


def dit_sp_a2a_counts(L: Layout, direction: int, nplanes: int, rank: int):
    U = L.raw.U
    arrs = [(c_int64 * U)() for _ in range(4)]
    check(lib().dit_sp_a2a_counts(byref(L.raw), direction, nplanes, rank, *arrs))
    return tuple(list(a) for a in arrs)


def dit_ulysses_pack(L: Layout, direction: int, srcs: Sequence[torch.Tensor], send: torch.Tensor,
                     stream=None) -> None:
    arr = (c_void_p * 3)(*[_addr(s) for s in srcs])
    check(lib().dit_ulysses_pack(byref(L.raw), direction, len(srcs), arr, _dt(srcs[0]),
                                 _ptr(send), _dt(send), _stream(stream)))


def dit_a2a_sim(L: Layout, direction: int, nplanes: int, send: torch.Tensor, recv: torch.Tensor,
                stream=None) -> None:
    check(lib().dit_a2a_sim(byref(L.raw), direction, nplanes, _ptr(send), _ptr(recv), _dt(send),
                            _stream(stream)))


def dit_sp_signal(L: Layout, arrival: torch.Tensor, epoch: int, ranks=None, stream=None) -> None:
    """Publish `epoch` on the arrival counters of `ranks` (all if None)."""
    mask = None
    if ranks is not None:
        n = L.raw.U * L.raw.R
        mask = (ctypes.c_ubyte * n)(*[1 if i in set(ranks) else 0 for i in range(n)])
    check(lib().dit_sp_signal(byref(L.raw), _ptr(arrival), mask, epoch & 0xFFFFFFFF, _stream(stream)))


def dit_a2a_sim_checked(L: Layout, direction: int, nplanes: int, send: torch.Tensor, recv: torch.Tensor,
                        arrival: torch.Tensor, epoch: int, timeout_ns: int,
                        status: Optional[torch.Tensor] = None, stream=None) -> None:
    check(lib().dit_a2a_sim_checked(byref(L.raw), direction, nplanes, _ptr(send), _ptr(recv), _dt(send),
                                    _ptr(arrival), epoch & 0xFFFFFFFF, int(timeout_ns), _ptr(status),
                                    _stream(stream)))


def dit_ulysses_unpack(L: Layout, direction: int, recv: torch.Tensor, dsts: Sequence[torch.Tensor],
                       range_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    ptrs = (c_void_p * 3)(*[_addr(d) for d in dsts])
    dts = (c_int * 3)(*[_dt(d) for d in dsts])
    check(lib().dit_ulysses_unpack(byref(L.raw), direction, len(dsts), _ptr(recv), _dt(recv), ptrs,
                                   dts, _ptr(range_flag), _stream(stream)))


def _ptrs(ts: Optional[Sequence[torch.Tensor]], n: int):
    return None if ts is None else (c_void_p * n)(*[_addr(t) for t in ts])


def dit_ulysses_pack_joint(L: Layout, txt: Optional[Sequence[torch.Tensor]], img: Optional[Sequence[torch.Tensor]],
                           send: torch.Tensor, stream=None) -> None:
    """Seq->head pack of the joint sequence [text; image]: txt[p] [B,S_txt,H,D],
    img[p] [B,S-S_txt,H,D] (either may be None when it has no rows)."""
    planes = txt if txt is not None else img
    n = len(planes)
    S_txt = txt[0].shape[1] if txt is not None else 0
    check(lib().dit_ulysses_pack_joint(byref(L.raw), n, _ptrs(txt, n), _ptrs(img, n), S_txt, _dt(planes[0]),
                                       _ptr(send), _dt(send), _stream(stream)))


def dit_ulysses_unpack_joint(L: Layout, recv: torch.Tensor, out_txt: Optional[torch.Tensor],
                             out_img: Optional[torch.Tensor], stream=None) -> None:
    """Head->seq unpack into the text rows (out_txt) and image rows (out_img)."""
    S_txt = out_txt.shape[1] if out_txt is not None else 0
    out = out_txt if out_txt is not None else out_img
    check(lib().dit_ulysses_unpack_joint(byref(L.raw), _ptr(recv), _dt(recv), _ptr(out_txt), _ptr(out_img),
                                         S_txt, _dt(out), _stream(stream)))


def dit_ulysses_unpack_rope(L: Layout, recv: torch.Tensor, dsts: Sequence[torch.Tensor], cos: torch.Tensor,
                            sin: torch.Tensor, rope_planes: int = 0x3,
                            range_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """Seq->head unpack that rotates the planes in rope_planes; cos/sin are
    float32 [S, D/2] tables of the joint sequence's positions."""
    for t in (cos, sin):
        if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != (L.raw.S, L.raw.D // 2):
            raise ValueError("rotary tables must be contiguous float32 [S, D/2]")
    ptrs = (c_void_p * 3)(*[_addr(d) for d in dsts])
    dts = (c_int * 3)(*[_dt(d) for d in dsts])
    check(lib().dit_ulysses_unpack_rope(byref(L.raw), len(dsts), _ptr(recv), _dt(recv), ptrs, dts, _ptr(cos),
                                        _ptr(sin), rope_planes, _ptr(range_flag), _stream(stream)))


def dit_ulysses_seq_to_head(L: Layout, srcs: Sequence[torch.Tensor], dsts: Sequence[torch.Tensor],
                            range_flag: Optional[torch.Tensor] = None, rope=None, rope_planes: int = 0x3,
                            src2: Optional[Sequence[torch.Tensor]] = None, stream=None) -> None:
    """Sequence layout -> head layout in one pass (pack, exchange and unpack
    composed): srcs[p] [B,S,H,D] -> dsts[p] [R,B,S_cap,Hp,D].  With src2,
    srcs[p] holds the first rows of the joint sequence ([B,split,H,D], e.g.
    the text stream) and src2[p] the rest ([B,S-split,H,D]).  rope: optional
    (cos, sin) float32 [S, D/2] tables; the planes in rope_planes are then
    rotated."""
    n = len(dsts)
    if len(srcs) != n or (src2 is not None and len(src2) != n):
        raise ValueError("one source (pair) per destination plane")
    split = srcs[0].shape[1] if src2 is not None else 0
    cos = sin = None
    planes = 0
    if rope is not None:
        cos, sin = rope
        for t in (cos, sin):
            if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != (L.raw.S, L.raw.D // 2):
                raise ValueError("rotary tables must be contiguous float32 [S, D/2]")
        planes = rope_planes
    dts = (c_int * 3)(*[_dt(d) for d in dsts])
    check(lib().dit_ulysses_seq_to_head(byref(L.raw), n, _ptrs(srcs, n), _ptrs(src2, n), split, _dt(srcs[0]),
                                        _ptrs(dsts, n), dts, _ptr(cos), _ptr(sin), planes, _ptr(range_flag),
                                        _stream(stream)))


def dit_ulysses_head_to_seq(L: Layout, src: torch.Tensor, dst: torch.Tensor, dst2: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    """Head layout [R,B,S_cap,Hp,D] -> sequence layout [B,S,H,D] in one pass.
    With dst2, dst takes the first rows of the joint sequence ([B,split,H,D])
    and dst2 the rest ([B,S-split,H,D])."""
    split = dst.shape[1] if dst2 is not None else 0
    check(lib().dit_ulysses_head_to_seq(byref(L.raw), _ptr(src), _dt(src), _ptr(dst), _ptr(dst2), split, _dt(dst),
                                        _stream(stream)))


def _view(t: torch.Tensor, kind: str) -> DitView:
    """kind: 'q' [n_q,B,S,H,D], 'kv' [n_kv,B,S,H,D], 'o' [n_q,n_kv,B,S,H,D],
    'out' [n_q,B,S,H,D], 'single' [B,S,H,D]."""
    st = t.stride()
    if st[-1] != 1:
        raise ValueError("the head dim must be contiguous")
    v = DitView()
    v.ptr = _addr(t)
    if kind in ("q", "out"):
        v.stride_q, v.stride_b, v.stride_s, v.stride_h = st[0], st[1], st[2], st[3]
    elif kind == "kv":
        v.stride_kv, v.stride_b, v.stride_s, v.stride_h = st[0], st[1], st[2], st[3]
    elif kind == "o":
        v.stride_q, v.stride_kv, v.stride_b, v.stride_s, v.stride_h = st[0], st[1], st[2], st[3], st[4]
    elif kind == "single":
        v.stride_b, v.stride_s, v.stride_h = st[0], st[1], st[2]
    elif kind == "packed":  # [T, H, D]
        v.stride_s, v.stride_h = st[0], st[1]
    else:
        raise ValueError(kind)
    return v


def _lse_view(t: Optional[torch.Tensor], kind: str) -> DitLseView:
    v = DitLseView()
    if t is None:
        return v
    if t.dtype != torch.float32 or t.stride(-1) != 1:
        raise ValueError("lse must be float32 with contiguous rows")
    st = t.stride()
    v.ptr = _addr(t)
    if kind == "o":        # [n_q, n_kv, B, H, S]
        v.stride_q, v.stride_kv, v.stride_b, v.stride_h = st[0], st[1], st[2], st[3]
    elif kind == "out":    # [n_q, B, H, S]
        v.stride_q, v.stride_b, v.stride_h = st[0], st[1], st[2]
    elif kind == "single":  # [B, H, S]
        v.stride_b, v.stride_h = st[0], st[1]
    elif kind == "packed":  # [H, T]
        v.stride_h = st[0]
    else:
        raise ValueError(kind)
    return v


def _lens(vals: Optional[Sequence[int]], n: int, default: int):
    vals = [default] * n if vals is None else list(vals)
    if len(vals) != n:
        raise ValueError("length list does not match the block count")
    return (c_int * max(n, 1))(*vals)


def dit_attn_partial(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                     lse: Optional[torch.Tensor] = None, q_len: Optional[Sequence[int]] = None,
                     kv_len: Optional[Sequence[int]] = None, scale: Optional[float] = None,
                     status: Optional[torch.Tensor] = None, stream=None) -> None:
    """All (query block, key/value block) partials in one launch."""
    n_q, B, Sq, H, D = q.shape
    n_kv = k.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    check(lib().dit_attn_partial(B, H, D, float(scale), n_q, _lens(q_len, n_q, Sq), n_kv,
                                 _lens(kv_len, n_kv, k.shape[2]), _view(q, "q"), _dt(q),
                                 _view(k, "kv"), _view(v, "kv"), _dt(v), _view(o, "o"), _dt(o),
                                 _lse_view(lse, "o"), _ptr(status), _stream(stream)))


def dit_attn_ring(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                  lse: Optional[torch.Tensor] = None, q_len: Optional[Sequence[int]] = None,
                  kv_len: Optional[Sequence[int]] = None, scale: Optional[float] = None,
                  status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Every query block against all key/value blocks, folded into one
    result per query block: q [n_q,B,S,H,D], k/v [n_kv,B,S,H,D],
    o [n_q,B,S,H,D], lse [n_q,B,H,S] (float32, optional)."""
    n_q, B, Sq, H, D = q.shape
    n_kv = k.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    check(lib().dit_attn_ring(B, H, D, float(scale), n_q, _lens(q_len, n_q, Sq), n_kv,
                              _lens(kv_len, n_kv, k.shape[2]), _view(q, "q"), _dt(q),
                              _view(k, "kv"), _view(v, "kv"), _dt(v), _view(o, "out"), _dt(o),
                              _lse_view(lse, "out"), _ptr(status), _stream(stream)))


def dit_attn_ring_rows(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                       o_row0: Sequence[int], lse: Optional[torch.Tensor] = None,
                       q_len: Optional[Sequence[int]] = None, kv_len: Optional[Sequence[int]] = None,
                       scale: Optional[float] = None, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """dit_attn_ring with every query block's output in one tensor o
    [B,S,H,D]: query block r's rows start at row o_row0[r]."""
    n_q, B, Sq, H, D = q.shape
    n_kv = k.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if len(o_row0) != n_q:
        raise ValueError("o_row0 needs one entry per query block")
    check(lib().dit_attn_ring_rows(B, H, D, float(scale), n_q, _lens(q_len, n_q, Sq), (c_int * n_q)(*o_row0), n_kv,
                                   _lens(kv_len, n_kv, k.shape[2]), _view(q, "q"), _dt(q),
                                   _view(k, "kv"), _view(v, "kv"), _dt(v), _view(o, "single"), _dt(o),
                                   _lse_view(lse, "out"), _ptr(status), _stream(stream)))


def dit_attn_ring_merge_static(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                               lse: Optional[torch.Tensor] = None, q_len: Optional[Sequence[int]] = None,
                               kv_len: Optional[Sequence[int]] = None, scale: Optional[float] = None,
                               status: Optional[torch.Tensor] = None, stream=None) -> None:
    """dit_attn_ring's arguments and result, computed as fp32 partials and
    their merge in the library's fixed device scratch array: the call
    allocates no memory, for callers that cannot.  Calls that overlap on the
    GPU share that array and race; the partials must fit
    DIT_RING_STATIC_SCRATCH_BYTES."""
    n_q, B, Sq, H, D = q.shape
    n_kv = k.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    check(lib().dit_attn_ring_merge_static(B, H, D, float(scale), n_q, _lens(q_len, n_q, Sq), n_kv,
                                           _lens(kv_len, n_kv, k.shape[2]), _view(q, "q"), _dt(q),
                                           _view(k, "kv"), _view(v, "kv"), _dt(v), _view(o, "out"), _dt(o),
                                           _lse_view(lse, "out"), _ptr(status), _stream(stream)))


def dit_attn_merge_lse(parts: torch.Tensor, lse_parts: torch.Tensor, out: torch.Tensor,
                       lse_out: Optional[torch.Tensor] = None,
                       q_len: Optional[Sequence[int]] = None, stream=None) -> None:
    n_q, n_parts, B, S, H, D = parts.shape
    check(lib().dit_attn_merge_lse(B, H, D, n_q, _lens(q_len, n_q, S), n_parts, _view(parts, "o"),
                                   _dt(parts), _lse_view(lse_parts, "o"), _view(out, "out"), _dt(out),
                                   _lse_view(lse_out, "out"), _stream(stream)))


def dit_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                  lse: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                  status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Single-shot attention: q [B,Sq,H,D], k/v [B,Sk,H,D], o [B,Sq,H,D]."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    check(lib().dit_attention(B, H, D, float(scale), Sq, Sk, _view(q, "single"), _dt(q),
                              _view(k, "single"), _view(v, "single"), _dt(v), _view(o, "single"),
                              _dt(o), _lse_view(lse, "single"), _ptr(status), _stream(stream)))


def dit_attn_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                    cu_q: Sequence[int], cu_k: Sequence[int], lse: Optional[torch.Tensor] = None,
                    scale: Optional[float] = None, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Packed variable-length attention: q, o [Tq, H, D]; k, v [Tk, H, D];
    sequence s has rows [cu_q[s], cu_q[s+1]) and keys [cu_k[s], cu_k[s+1]);
    lse [H, Tq] (float32) optional."""
    _, H, D = q.shape
    n = len(cu_q) - 1
    if len(cu_k) != n + 1 or n < 0:
        raise ValueError("cu_q and cu_k need the same number of sequences")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    cq = (c_int * max(n + 1, 1))(*cu_q)
    ck = (c_int * max(n + 1, 1))(*cu_k)
    check(lib().dit_attn_varlen(H, D, float(scale), n, cq, ck, _view(q, "packed"), _dt(q), _view(k, "packed"),
                                _view(v, "packed"), _dt(v), _view(o, "packed"), _dt(o), _lse_view(lse, "packed"),
                                _ptr(status), _stream(stream)))


def dit_cfg_combine(pred: torch.Tensor, out: torch.Tensor, g: float, stream=None) -> None:
    """pred [2, ...] (0 = unconditional, 1 = conditional) -> out [...]."""
    if not (pred.is_contiguous() and out.is_contiguous()):
        raise ValueError("cfg combine needs contiguous tensors")
    N = out.numel()
    if pred.numel() != 2 * N:
        raise ValueError("pred must hold two branches of out's size")
    check(lib().dit_cfg_combine(_ptr(pred), _dt(pred), N, float(g), _ptr(out), _dt(out),
                                _stream(stream)))


def dit_device_status(reset: bool = True) -> int:
    code = c_int(0)
    check(lib().dit_device_status(byref(code), 1 if reset else 0))
    return code.value
