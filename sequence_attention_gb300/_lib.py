"""ctypes declarations of libditsp.so (the C ABI in include/ditsp.h).

Loading fails loudly: there is no fallback implementation.  Build the
library with ``python sequence_attention_gb300/build.py`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, Structure, c_char_p, c_float, c_int, c_int64, c_uint, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libditsp.so")

DIT_MAX_U = 64
DIT_MAX_R = 8
DIT_MAX_RANKS = 64
#: bytes of the fixed device scratch array of dit_attn_ring_merge_static
DIT_RING_STATIC_SCRATCH_BYTES = 64 * 1024 * 1024

DIT_OK, DIT_ERR_INVALID_ARG, DIT_ERR_UNSUPPORTED, DIT_ERR_CUDA, DIT_ERR_TIMEOUT, DIT_ERR_RANGE = range(6)
DIT_F32, DIT_BF16, DIT_F16, DIT_E4M3 = range(4)
DIT_LAYOUT_NOPAD_HEADS, DIT_LAYOUT_PAD_LCM64 = 1, 2
DIT_SEQ_TO_HEAD, DIT_HEAD_TO_SEQ = range(2)

#: every function include/ditsp.h declares
EXPORTS = (
    "dit_status_string", "dit_last_error", "dit_device_status", "dit_sp_layout_init", "dit_sp_layout_init_ex",
    "dit_sp_a2a_counts", "dit_ulysses_pack", "dit_a2a_sim", "dit_ulysses_unpack",
    "dit_attn_partial", "dit_attn_merge_lse", "dit_attention", "dit_cfg_combine",
    "dit_sp_signal", "dit_a2a_sim_checked", "dit_ulysses_pack_joint", "dit_ulysses_unpack_joint",
    "dit_ulysses_unpack_rope", "dit_attn_varlen", "dit_ulysses_seq_to_head", "dit_ulysses_head_to_seq",
    "dit_attn_ring",
    "dit_attn_ring_rows",
    "dit_attn_ring_merge_static",
)


class DitSpLayout(Structure):
    _fields_ = [(n, c_int) for n in ("B", "S", "H", "D", "U", "R", "Hp", "Hl", "S_cap")] + [
        ("ring_len", c_int * DIT_MAX_R),
        ("ring_off", c_int * DIT_MAX_R),
        ("rank_len", c_int * DIT_MAX_RANKS),
        ("rank_off", c_int * DIT_MAX_RANKS),
        ("S_pad", c_int),
        ("flags", c_int),
        ("head_len", c_int * DIT_MAX_U),
        ("head_off", c_int * DIT_MAX_U),
        ("ring_real", c_int * DIT_MAX_R),
    ]


class DitView(Structure):
    _fields_ = [("ptr", c_void_p)] + [(n, c_int64) for n in
                                      ("stride_q", "stride_kv", "stride_b", "stride_s", "stride_h")]


class DitLseView(Structure):
    _fields_ = [("ptr", c_void_p)] + [(n, c_int64) for n in
                                      ("stride_q", "stride_kv", "stride_b", "stride_h")]


class DitError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{status_name(status)}: {msg}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python sequence_attention_gb300/build.py`")
    L = ctypes.CDLL(LIB_PATH)
    L.dit_status_string.restype = c_char_p
    L.dit_status_string.argtypes = [c_int]
    L.dit_last_error.restype = c_char_p
    L.dit_last_error.argtypes = []
    L.dit_device_status.restype = c_int
    L.dit_device_status.argtypes = [POINTER(c_int), c_int]
    L.dit_sp_layout_init.restype = c_int
    L.dit_sp_layout_init.argtypes = [c_int] * 6 + [POINTER(DitSpLayout)]
    L.dit_sp_layout_init_ex.restype = c_int
    L.dit_sp_layout_init_ex.argtypes = [c_int] * 7 + [POINTER(DitSpLayout)]
    L.dit_sp_a2a_counts.restype = c_int
    L.dit_sp_a2a_counts.argtypes = [POINTER(DitSpLayout), c_int, c_int, c_int] + [POINTER(c_int64)] * 4
    L.dit_ulysses_pack.restype = c_int
    L.dit_ulysses_pack.argtypes = [POINTER(DitSpLayout), c_int, c_int, POINTER(c_void_p), c_int,
                                   c_void_p, c_int, c_void_p]
    L.dit_a2a_sim.restype = c_int
    L.dit_a2a_sim.argtypes = [POINTER(DitSpLayout), c_int, c_int, c_void_p, c_void_p, c_int, c_void_p]
    L.dit_sp_signal.restype = c_int
    L.dit_sp_signal.argtypes = [POINTER(DitSpLayout), c_void_p, c_void_p, c_uint, c_void_p]
    L.dit_a2a_sim_checked.restype = c_int
    L.dit_a2a_sim_checked.argtypes = [POINTER(DitSpLayout), c_int, c_int, c_void_p, c_void_p, c_int, c_void_p,
                                      c_uint, c_int64, c_void_p, c_void_p]
    L.dit_ulysses_unpack.restype = c_int
    L.dit_ulysses_unpack.argtypes = [POINTER(DitSpLayout), c_int, c_int, c_void_p, c_int,
                                     POINTER(c_void_p), POINTER(c_int), c_void_p, c_void_p]
    L.dit_ulysses_pack_joint.restype = c_int
    L.dit_ulysses_pack_joint.argtypes = [POINTER(DitSpLayout), c_int, POINTER(c_void_p), POINTER(c_void_p),
                                         c_int, c_int, c_void_p, c_int, c_void_p]
    L.dit_ulysses_unpack_joint.restype = c_int
    L.dit_ulysses_unpack_joint.argtypes = [POINTER(DitSpLayout), c_void_p, c_int, c_void_p, c_void_p, c_int,
                                           c_int, c_void_p]
    L.dit_ulysses_unpack_rope.restype = c_int
    L.dit_ulysses_unpack_rope.argtypes = [POINTER(DitSpLayout), c_int, c_void_p, c_int, POINTER(c_void_p),
                                          POINTER(c_int), c_void_p, c_void_p, c_uint, c_void_p, c_void_p]
    L.dit_ulysses_seq_to_head.restype = c_int
    L.dit_ulysses_seq_to_head.argtypes = [POINTER(DitSpLayout), c_int, POINTER(c_void_p), POINTER(c_void_p), c_int,
                                          c_int, POINTER(c_void_p), POINTER(c_int), c_void_p, c_void_p, c_uint,
                                          c_void_p, c_void_p]
    L.dit_ulysses_head_to_seq.restype = c_int
    L.dit_ulysses_head_to_seq.argtypes = [POINTER(DitSpLayout), c_void_p, c_int, c_void_p, c_void_p, c_int, c_int,
                                          c_void_p]
    L.dit_attn_partial.restype = c_int
    L.dit_attn_partial.argtypes = [c_int, c_int, c_int, c_float, c_int, POINTER(c_int), c_int,
                                   POINTER(c_int), DitView, c_int, DitView, DitView, c_int, DitView,
                                   c_int, DitLseView, c_void_p, c_void_p]
    L.dit_attn_ring.restype = c_int
    L.dit_attn_ring.argtypes = [c_int, c_int, c_int, c_float, c_int, POINTER(c_int), c_int,
                                POINTER(c_int), DitView, c_int, DitView, DitView, c_int, DitView,
                                c_int, DitLseView, c_void_p, c_void_p]
    L.dit_attn_ring_rows.restype = c_int
    L.dit_attn_ring_rows.argtypes = [c_int, c_int, c_int, c_float, c_int, POINTER(c_int), POINTER(c_int), c_int,
                                     POINTER(c_int), DitView, c_int, DitView, DitView, c_int, DitView,
                                     c_int, DitLseView, c_void_p, c_void_p]
    L.dit_attn_ring_merge_static.restype = c_int
    L.dit_attn_ring_merge_static.argtypes = [c_int, c_int, c_int, c_float, c_int, POINTER(c_int), c_int,
                                             POINTER(c_int), DitView, c_int, DitView, DitView, c_int, DitView,
                                             c_int, DitLseView, c_void_p, c_void_p]
    L.dit_attn_varlen.restype = c_int
    L.dit_attn_varlen.argtypes = [c_int, c_int, c_float, c_int, POINTER(c_int), POINTER(c_int), DitView, c_int,
                                  DitView, DitView, c_int, DitView, c_int, DitLseView, c_void_p, c_void_p]
    L.dit_attn_merge_lse.restype = c_int
    L.dit_attn_merge_lse.argtypes = [c_int, c_int, c_int, c_int, POINTER(c_int), c_int, DitView, c_int,
                                     DitLseView, DitView, c_int, DitLseView, c_void_p]
    L.dit_attention.restype = c_int
    L.dit_attention.argtypes = [c_int, c_int, c_int, c_float, c_int, c_int, DitView, c_int, DitView,
                                DitView, c_int, DitView, c_int, DitLseView, c_void_p, c_void_p]
    L.dit_cfg_combine.restype = c_int
    L.dit_cfg_combine.argtypes = [c_void_p, c_int, c_int64, c_float, c_void_p, c_int, c_void_p]
    _lib = L
    return L


def status_name(s: int) -> str:
    names = {0: "DIT_OK", 1: "DIT_ERR_INVALID_ARG", 2: "DIT_ERR_UNSUPPORTED", 3: "DIT_ERR_CUDA",
             4: "DIT_ERR_TIMEOUT", 5: "DIT_ERR_RANGE"}
    return names.get(s, f"DIT_ERR_{s}")


def check(status: int) -> None:
    if status != DIT_OK:
        raise DitError(status, lib().dit_last_error().decode(errors="replace"))
