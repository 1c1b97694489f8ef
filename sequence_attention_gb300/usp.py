"""Unified sequence parallelism (Ulysses inside, ring outside) on one GPU.

The U*R virtual ranks are partitions of the buffers below, all in one GPU's
memory; every step is one call into libditsp (cache-dit "Context
Parallelism", USP: Ulysses all-to-all, then ring attention on the
redistributed data, then the inverse all-to-all; SGLang Diffusion
"Parallelism Overview", What happens to the shapes):

  layout in    seq-sharded Q,K,V -> head layout [R,B,S_cap,Hp,D] (V as f16)
  attention    every ring block r against every ring block j, one launch:
               ring_merge="fold" (default on 16-bit inputs) dit_attn_ring, each hop folded in
               by the online softmax as the kernel walks the K/V blocks;
               ring_merge="partials" dit_attn_partial (every (r, j)
               partial) then dit_attn_merge_lse (the R-way log-sum-exp
               merge), the form whose partials could come from other GPUs
  layout out   head layout -> seq-sharded output [B,S,H,D]; with the
               one-pass exchange and one result per query block (R = 1 or
               the fold) the attention writes each block's rows straight to
               their sequence positions (dit_attn_ring_rows) and this pass
               is skipped

The layout steps run one of two ways (``exchange``):
  "direct"  dit_ulysses_seq_to_head / dit_ulysses_head_to_seq: on one memory
            the exchange aliases receive and send blocks, so pack, exchange
            and unpack are one pass (each element read and written once);
  "a2a"     dit_ulysses_pack -> dit_a2a_sim -> dit_ulysses_unpack, the three
            calls a multi-GPU build keeps (the exchange becomes an alltoallv
            with the counts of dit_sp_a2a_counts); the e4m3 wire needs it.
Both give the same bits.

With rotary tables, the seq-to-head step is the receive preparation that
rotates Q and K as it writes them; run_joint() takes the paired text and
image streams of a double-stream block and returns the output in the same
two streams, so the joint sequence is never concatenated.

All buffers are allocated once, when the plan is built; run() allocates
nothing and only enqueues kernels on the current (or given) stream.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence, Tuple

import torch

from . import (DIT_HEAD_TO_SEQ, DIT_SEQ_TO_HEAD, DitError, dit_a2a_sim, dit_attn_merge_lse, dit_attn_partial,
               dit_attn_ring, dit_attn_ring_rows,
               dit_sp_layout_init, dit_ulysses_head_to_seq, dit_ulysses_pack, dit_ulysses_pack_joint,
               dit_ulysses_seq_to_head, dit_ulysses_unpack, dit_ulysses_unpack_joint, dit_ulysses_unpack_rope)
from ._lib import DIT_ERR_RANGE, DIT_ERR_TIMEOUT


class UspPlan:
    def __init__(self, B: int, S: int, H: int, D: int, U: int, R: int,
                 in_dtype: torch.dtype = torch.bfloat16,
                 out_dtype: Optional[torch.dtype] = None,
                 v_dtype: Optional[torch.dtype] = None,
                 device: str = "cuda", scale: Optional[float] = None,
                 rope: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
                 fp8_qv: bool = False, fp8_o: bool = False,
                 pad_heads: bool = True, pad_lcm64: bool = False,
                 parts_dtype: Optional[torch.dtype] = None, exchange: Optional[str] = None,
                 ring_merge: Optional[str] = None):
        """rope: optional (cos, sin) float32 [S, D/2] device tables of the
        joint sequence; Q and K are then rotated by the receive preparation.
        fp8_qv / fp8_o: Q and V (one exchange) / the output cross the
        all-to-all as e4m3 records; K keeps its own 16-bit exchange.
        pad_heads=False: uneven head groups without padding; pad_lcm64: the
        sequence padded to a multiple of lcm(U*R, 64), padding rows excluded
        from attention.
        parts_dtype: type of the R x R ring partials (R > 1).  By default f16
        when V is f16 and the output 16-bit: a partial is a convex
        combination of V rows, so it stays within V's range, and f16 keeps
        11 significant bits against the output's 8 (bf16), at half the
        bytes of f32 for the attention's stores and the merge's loads.
        Otherwise f32.
        ring_merge: "fold" (the K/V blocks folded into one result as the
        kernel walks them) or "partials" (every partial written, then the
        R-way merge kernel); the same result up to rounding.  By default
        "fold" on 16-bit inputs and "partials" on the fp32 path: measured
        on one GB300, the fold saves the merge pass and the partials' writes
        (FLUX-1008-like R = 2: 0.246 against 0.266 ms per step; Wan-like
        R = 4: 79.1 against 80.8 ms), while the fp32 CUDA-core kernel folds
        with half the CTAs of its partials (tiny: 0.116 against 0.106 ms).
        exchange: "direct" (one pass per layout step) or "a2a" (pack,
        exchange, unpack); default "direct", or "a2a" with an e4m3 wire.
        v_dtype: by default f16 for bf16 inputs (P V runs with P in V's type,
        and f16 keeps P to 11 significant bits).  f16 holds |v| < 65520: a
        larger V value becomes infinite and makes the output inf/NaN.  The
        layout step then sets the plan's range flag; check() reports it.  Pass
        v_dtype=torch.bfloat16 for inputs that may exceed that range."""
        self.L = dit_sp_layout_init(B, S, H, D, U, R, pad_heads, pad_lcm64)
        self.B, self.S, self.H, self.D, self.U, self.R = B, S, H, D, U, R
        self.in_dtype = in_dtype
        self.wire_dtype = in_dtype
        self.out_dtype = out_dtype or in_dtype
        if v_dtype is None:
            # P V runs with P in V's type: f16 keeps P to 11 significant bits,
            # which keeps the ring merge within 1e-3 of single-shot attention
            v_dtype = torch.float16 if in_dtype == torch.bfloat16 else in_dtype
        self.v_dtype = v_dtype
        self.scale = 1.0 / math.sqrt(D) if scale is None else scale
        L = self.L
        hs = L.head_shape()
        dev = torch.device(device)
        self.fp8_qv, self.fp8_o = fp8_qv, fp8_o
        if exchange is None:
            exchange = "a2a" if (fp8_qv or fp8_o) else "direct"
        if exchange not in ("direct", "a2a"):
            raise ValueError(f"exchange must be 'direct' or 'a2a', got {exchange!r}")
        if exchange == "direct" and (fp8_qv or fp8_o):
            raise ValueError("the e4m3 wire needs exchange='a2a' (the direct path has no wire)")
        self.exchange = exchange
        direct = exchange == "direct"
        self.send = self.recv = self.send_qv = self.recv_qv = self.send_o = self.recv_o = None
        if direct:
            pass
        elif fp8_qv:
            self.send_qv = torch.empty(L.wire_bytes_e4m3(2), dtype=torch.uint8, device=dev)
            self.recv_qv = torch.empty_like(self.send_qv)
            self.send = torch.empty(L.wire_elems(1), dtype=in_dtype, device=dev)     # K
        else:
            self.send = torch.empty(L.wire_elems(3), dtype=in_dtype, device=dev)
        if not direct:
            self.recv = torch.empty_like(self.send)
        self.q_h = torch.empty(hs, dtype=in_dtype, device=dev)
        self.k_h = torch.empty(hs, dtype=in_dtype, device=dev)
        self.v_h = torch.empty(hs, dtype=v_dtype, device=dev)
        self.o_h = torch.empty(hs, dtype=self.out_dtype, device=dev)
        if parts_dtype is None:
            half_ok = v_dtype == torch.float16 and self.out_dtype in (torch.bfloat16, torch.float16)
            parts_dtype = torch.float16 if half_ok else torch.float32
        if parts_dtype == torch.float16 and v_dtype != torch.float16:
            raise ValueError("f16 partials need f16 V (a partial lies within V's range)")
        self.parts_dtype = parts_dtype
        if ring_merge is None:
            ring_merge = "fold" if in_dtype != torch.float32 else "partials"
        if ring_merge not in ("fold", "partials"):
            raise ValueError(f"ring_merge must be 'fold' or 'partials', got {ring_merge!r}")
        self.ring_merge = ring_merge
        if R > 1 and ring_merge == "partials":
            self.parts = torch.empty((R, R) + tuple(hs[1:]), dtype=parts_dtype, device=dev)
            self.lse_parts = torch.empty((R, R, B, L.Hp, L.S_cap), dtype=torch.float32, device=dev)
        else:
            self.parts = self.lse_parts = None
        if direct:
            pass
        elif fp8_o:
            self.send_o = torch.empty(L.wire_bytes_e4m3(1), dtype=torch.uint8, device=dev)
        else:
            self.send_o = torch.empty(L.wire_elems(1), dtype=self.out_dtype, device=dev)
        if not direct:
            self.recv_o = torch.empty_like(self.send_o)
        self.rope = rope
        # device words the kernels set and never clear: [0] the range flag of
        # the layout step (a value that overflowed its 16-bit destination),
        # [1] the attention's status (a bounded wait that ran out)
        self.flags = torch.zeros(2, dtype=torch.int32, device=dev)
        self.range_flag = self.flags[0:1]
        self.status = self.flags[1:2]

    # ---- views of the real (unpadded) heads --------------------------------
    def heads(self, t: torch.Tensor) -> torch.Tensor:
        return t[..., : self.H, :]

    @property
    def ring_len(self):
        """Real (non-padding) rows of each ring block: the attention's
        query and key counts (the layout's ring_real)."""
        return self.L.ring_real

    def check(self, reset: bool = True) -> None:
        """Wait for the stream, then raise DitError if a kernel of an earlier
        run set the range flag (a value overflowed its 16-bit destination,
        e.g. |V| >= 65520 converted to f16) or the status word (a bounded wait
        ran out).  The words are sticky: they keep a set value across runs
        until this call (reset=True) clears them."""
        torch.cuda.current_stream(self.flags.device).synchronize()
        rng, st = (int(x) for x in self.flags.tolist())
        if reset and (rng or st):
            self.flags.zero_()
        if st:
            raise DitError(DIT_ERR_TIMEOUT if st == DIT_ERR_TIMEOUT else st,
                           "a bounded device-side wait ran out in the attention")
        if rng:
            raise DitError(DIT_ERR_RANGE, "a value overflowed its 16-bit destination type "
                                          "(f16 holds |x| < 65520; use v_dtype=torch.bfloat16)")

    def direct_out(self, out: torch.Tensor) -> bool:
        """Whether the attention can write `out` [B,S,H,D] in place of the
        layout-out pass: on one memory the head-to-sequence permutation only
        moves ring block r's rows to rows ring_off[r] + i and drops padded
        heads, so the attention's output view can do it, when it gives one
        result per query block (R = 1 or the fold) and out has the plan's
        shape in a type the attention writes."""
        if self.exchange != "direct" or not (self.R == 1 or self.ring_merge == "fold"):
            return False
        if tuple(out.shape) != (self.B, self.S, self.H, self.D) or out.stride(-1) != 1:
            return False
        return self.in_dtype != torch.float32 or out.dtype == torch.float32

    def steps(self):
        """Names of the kernels one run() launches, in order (run() with an
        output the attention can write in place)."""
        if self.exchange == "direct":
            s = ["seq_to_head"]
        elif self.fp8_qv:
            s = ["pack_s2h_k", "pack_s2h_qv", "a2a_s2h_k", "a2a_s2h_qv", "unpack_s2h_k", "unpack_s2h_qv"]
        else:
            s = ["pack_s2h", "a2a_s2h", "unpack_s2h"]
        if self.R > 1 and self.ring_merge == "fold":
            s = s + ["attn_ring"]
        else:
            s = s + ["attn_partial"]
            if self.R > 1:
                s.append("merge")
        if self.exchange != "direct":
            return s + ["pack_h2s", "a2a_h2s", "unpack_h2s"]
        return s if (self.R == 1 or self.ring_merge == "fold") else s + ["head_to_seq"]

    def _unpack(self, recv, heads, rope_mask, stream):
        if self.rope is not None:
            dit_ulysses_unpack_rope(self.L, recv, heads, self.rope[0], self.rope[1], rope_mask,
                                    self.range_flag, stream)
        else:
            dit_ulysses_unpack(self.L, DIT_SEQ_TO_HEAD, recv, heads, self.range_flag, stream)

    def _receive(self, stream):
        L = self.L
        if self.fp8_qv:
            dit_a2a_sim(L, DIT_SEQ_TO_HEAD, 1, self.send, self.recv, stream)
            dit_a2a_sim(L, DIT_SEQ_TO_HEAD, 2, self.send_qv, self.recv_qv, stream)
            self._unpack(self.recv, [self.k_h], 0b1, stream)
            self._unpack(self.recv_qv, [self.q_h, self.v_h], 0b01, stream)
        else:
            dit_a2a_sim(L, DIT_SEQ_TO_HEAD, 3, self.send, self.recv, stream)
            self._unpack(self.recv, [self.q_h, self.k_h, self.v_h], 0b011, stream)

    def layout_in(self, q, k, v, stream=None):
        if self.exchange == "direct":
            dit_ulysses_seq_to_head(self.L, [q, k, v], [self.q_h, self.k_h, self.v_h], self.range_flag,
                                    rope=self.rope, rope_planes=0b011, stream=stream)
            return
        if self.fp8_qv:
            dit_ulysses_pack(self.L, DIT_SEQ_TO_HEAD, [k], self.send, stream)
            dit_ulysses_pack(self.L, DIT_SEQ_TO_HEAD, [q, v], self.send_qv, stream)
        else:
            dit_ulysses_pack(self.L, DIT_SEQ_TO_HEAD, [q, k, v], self.send, stream)
        self._receive(stream)

    def layout_in_joint(self, txt: Optional[Sequence[torch.Tensor]], img: Optional[Sequence[torch.Tensor]],
                        stream=None):
        """txt / img: (q, k, v) of the text [B,S_txt,H,D] and image
        [B,S-S_txt,H,D] streams (None for a stream without rows)."""
        if self.exchange == "direct":
            first, second = (txt, img) if txt is not None else (img, None)
            dit_ulysses_seq_to_head(self.L, list(first), [self.q_h, self.k_h, self.v_h], self.range_flag,
                                    rope=self.rope, rope_planes=0b011,
                                    src2=None if second is None else list(second), stream=stream)
            return
        if self.fp8_qv:
            sel = lambda t, idx: None if t is None else [t[i] for i in idx]   # noqa: E731
            dit_ulysses_pack_joint(self.L, sel(txt, [1]), sel(img, [1]), self.send, stream)
            dit_ulysses_pack_joint(self.L, sel(txt, [0, 2]), sel(img, [0, 2]), self.send_qv, stream)
        else:
            dit_ulysses_pack_joint(self.L, txt, img, self.send, stream)
        self._receive(stream)

    def partials(self, stream=None, out: Optional[torch.Tensor] = None):
        """The attention of every ring block against every ring block in one
        launch: folded into the output (ring_merge="fold"), or every (r, j)
        partial written for merge(); with R = 1 the single partial is the
        output itself.  Given out (the step's [B,S,H,D] output) and
        direct_out(out), the result goes straight to out and layout_out(out)
        has nothing left to do."""
        rl = self.ring_len
        qv, kv, vv = self.heads(self.q_h), self.heads(self.k_h), self.heads(self.v_h)
        direct = out is not None and self.direct_out(out)
        self._o_at = out if direct else None
        if self.R == 1:
            o = (out if direct else self.heads(self.o_h)[0]).unsqueeze(0).unsqueeze(0)   # [1, 1, B, S, H, D]
            dit_attn_partial(qv, kv, vv, o, None, rl, rl, self.scale, self.status, stream)
        elif self.ring_merge == "fold" and direct:
            dit_attn_ring_rows(qv, kv, vv, out, self.L.ring_off, None, rl, rl, self.scale, self.status, stream)
        elif self.ring_merge == "fold":
            dit_attn_ring(qv, kv, vv, self.heads(self.o_h), None, rl, rl, self.scale, self.status, stream)
        else:
            dit_attn_partial(qv, kv, vv, self.heads(self.parts),
                             self.lse_parts[:, :, :, : self.H, :], rl, rl, self.scale,
                             self.status, stream)

    def merge(self, stream=None):
        """The ring's log-sum-exp merge of the R partials (nothing when R = 1
        or when the attention folded the blocks itself)."""
        if self.R > 1 and self.ring_merge == "partials":
            dit_attn_merge_lse(self.heads(self.parts), self.lse_parts[:, :, :, : self.H, :],
                               self.heads(self.o_h), None, self.ring_len, stream)

    def attend(self, stream=None, out: Optional[torch.Tensor] = None):
        self.partials(stream, out)
        self.merge(stream)

    def layout_out(self, out, stream=None):
        L = self.L
        if getattr(self, "_o_at", None) is out:
            return                      # the attention wrote out in place
        if self.exchange == "direct":
            dit_ulysses_head_to_seq(L, self.o_h, out, stream=stream)
            return
        dit_ulysses_pack(L, DIT_HEAD_TO_SEQ, [self.o_h], self.send_o, stream)
        dit_a2a_sim(L, DIT_HEAD_TO_SEQ, 1, self.send_o, self.recv_o, stream)
        dit_ulysses_unpack(L, DIT_HEAD_TO_SEQ, self.recv_o, [out], None, stream)

    def layout_out_joint(self, out_txt, out_img, stream=None):
        L = self.L
        if self.exchange == "direct":
            first, second = (out_txt, out_img) if out_txt is not None else (out_img, None)
            dit_ulysses_head_to_seq(L, self.o_h, first, second, stream=stream)
            return
        dit_ulysses_pack(L, DIT_HEAD_TO_SEQ, [self.o_h], self.send_o, stream)
        dit_a2a_sim(L, DIT_HEAD_TO_SEQ, 1, self.send_o, self.recv_o, stream)
        dit_ulysses_unpack_joint(L, self.recv_o, out_txt, out_img, stream)

    def run_joint(self, txt, img, out_txt, out_img, stream=None):
        """The double-stream block's attention: paired streams in and out."""
        self.layout_in_joint(txt, img, stream)
        self.attend(stream)
        self.layout_out_joint(out_txt, out_img, stream)

    def capture(self, q, k, v, out, extra=None):
        """A CUDA graph of run(q, k, v, out) (and of extra(), a callable that
        enqueues more calls, e.g. the CFG combine) for these tensors: replay()
        launches the whole step at once.  Every call of the step is a
        stream-ordered kernel launch and nothing is allocated, so the replay
        gives the same bits as run()."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.q_h.device)
        s.wait_stream(torch.cuda.current_stream(self.q_h.device))
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.run(q, k, v, out)
                if extra is not None:
                    extra()
        torch.cuda.current_stream(self.q_h.device).wait_stream(s)
        return g

    def run(self, q, k, v, out, stream=None, check: bool = False):
        """q, k, v: [B, S, H, D] seq-sharded inputs; out: [B, S, H, D].
        check=True waits for the step and raises as check() does."""
        self.layout_in(q, k, v, stream)
        self.attend(stream, out)
        self.layout_out(out, stream)
        if check:
            self.check()
        return out
