"""dit_attn_ring_merge_static: the ring's partials and merge with the
partials in the library's fixed device array, for callers that cannot
allocate device memory (an engine whose memory pool owns the device, or a
latency-critical path that must not stall on cudaMalloc/cudaFree).

The GPU test makes two calls in a row on one stream, of different shapes, so
the second runs on an array that still holds the first call's partials.  Each
result is checked against the library's existing calls on caller-allocated
buffers: dit_attn_partial into fp32 partials followed by dit_attn_merge_lse
(the same arithmetic), and the folded dit_attn_ring, both within the bar the
merge tests hold (relative RMS 1e-3; log-sum-exp within 1e-4).  This file is
named to be collected last.
"""
import numpy as np
import pytest
import torch

import synth
from tests.helpers import LSE_ABS, MERGE_REL_RMS, f64, max_abs, rel_rms


def _blocks(x, lens, cap):
    """[B, sum(lens), H, D] -> [n, B, cap, H, D] blocks, zero past each length."""
    B, _, H, D = x.shape
    out = torch.zeros((len(lens), B, cap, H, D), dtype=x.dtype)
    off = 0
    for j, n in enumerate(lens):
        out[j, :, :n] = x[:, off:off + n]
        off += n
    return out


def _inputs(B, H, D, q_lens, kv_lens, seed):
    Sq, Sk = sum(q_lens), sum(kv_lens)
    q = synth.normal((B, Sq, H, D), seed, 0.5, "bf16")
    k = synth.normal((B, max(Sk, 1), H, D), seed + 1, 0.5, "bf16")[:, :Sk]
    v = synth.normal((B, max(Sk, 1), H, D), seed + 2, 0.5, "bf16")
    cq, ck = max(q_lens), max(max(kv_lens), 1)
    return (_blocks(q, q_lens, cq).cuda(), _blocks(k, kv_lens, ck).cuda(),
            _blocks(v.to(torch.float16)[:, :Sk], kv_lens, ck).cuda())


def _check(got, ref, lse_got, lse_ref, q_lens, what):
    for r, n in enumerate(q_lens):
        g, e = f64(got[r, :, :n]), f64(ref[r, :, :n])
        assert np.all(np.isfinite(g)), f"{what}: non-finite output"
        rr = rel_rms(g, e)
        assert rr <= MERGE_REL_RMS, f"{what}: block {r} rel-RMS {rr:.3e}"
        lg, le = f64(lse_got[r, :, :, :n]), f64(lse_ref[r, :, :, :n])
        assert np.array_equal(np.isinf(lg), np.isinf(le)), f"{what}: block {r} lse -inf rows differ"
        fin = np.isfinite(le)
        assert max_abs(lg[fin], le[fin]) <= LSE_ABS, f"{what}: block {r} lse"


@pytest.mark.gpu
def test_static_scratch_matches_caller_buffers_twice():
    import sequence_attention_gb300 as sa
    calls = [
        # B, H, D, query block lengths, key block lengths, seed
        (1, 3, 128, [1121, 1120], [1121, 1120], 300),     # a FLUX-1008-like ring pair, three heads
        (2, 2, 64, [300, 5, 129], [128, 0, 77, 1], 310),  # ragged blocks, an empty and a one-key block
    ]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for B, H, D, q_lens, kv_lens, seed in calls:
        q, k, v = _inputs(B, H, D, q_lens, kv_lens, seed)
        n_q, n_kv, cq = len(q_lens), len(kv_lens), max(q_lens)
        out = torch.full((n_q, B, cq, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((n_q, B, H, cq), float("nan"), dtype=torch.float32, device="cuda")
        sa.dit_attn_ring_merge_static(q, k, v, out, lse, q_lens, kv_lens, status=status)

        parts = torch.empty((n_q, n_kv, B, cq, H, D), dtype=torch.float32, device="cuda")
        lse_parts = torch.empty((n_q, n_kv, B, H, cq), dtype=torch.float32, device="cuda")
        sa.dit_attn_partial(q, k, v, parts, lse_parts, q_lens, kv_lens, status=status)
        ref = torch.full_like(out, float("nan"))
        lse_ref = torch.full_like(lse, float("nan"))
        sa.dit_attn_merge_lse(parts, lse_parts, ref, lse_ref, q_lens)

        fold = torch.full_like(out, float("nan"))
        lse_fold = torch.full_like(lse, float("nan"))
        sa.dit_attn_ring(q, k, v, fold, lse_fold, q_lens, kv_lens, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _check(out, ref, lse, lse_ref, q_lens, f"partials+merge, B={B} H={H} D={D}")
        _check(out, fold, lse, lse_fold, q_lens, f"folded ring, B={B} H={H} D={D}")


def _call_host_only(B, H, D, q_lens, kv_lens):
    """Call the entry point with NULL tensors; only host-side checks run."""
    from ctypes import c_int

    from sequence_attention_gb300 import _lib
    L = _lib.lib()
    ql, kl = (c_int * len(q_lens))(*q_lens), (c_int * len(kv_lens))(*kv_lens)
    view, lse = _lib.DitView(), _lib.DitLseView()
    view.stride_s, view.stride_h = H * D, D                # [blocks][B][rows][H][D] rows of empty tensors
    st = L.dit_attn_ring_merge_static(B, H, D, 0.088, len(q_lens), ql, len(kv_lens), kl, view, _lib.DIT_BF16,
                                      view, view, _lib.DIT_F16, view, _lib.DIT_BF16, lse, None, None)
    return st, L.dit_last_error()


@pytest.mark.parametrize("B,H,D,q_lens", [
    (1, 24, 128, [4608, 4608]),              # FLUX-sized blocks: about 218 MiB of partials
    (1 << 30, 1 << 30, 128, [1 << 30] * 8),  # a size whose byte count would wrap 64 bits
    (1, 1, 1 << 30, [1 << 30]),
])
def test_static_scratch_rejects_a_request_beyond_its_size(B, H, D, q_lens):
    """Refused with DIT_ERR_INVALID_ARG before any device work (no GPU
    needed)."""
    from sequence_attention_gb300 import _lib
    rows = len(q_lens) * len(q_lens) * B * H * max(q_lens)
    assert rows * (4 * D + 4) > _lib.DIT_RING_STATIC_SCRATCH_BYTES
    st, msg = _call_host_only(B, H, D, q_lens, q_lens)
    assert st == _lib.DIT_ERR_INVALID_ARG
    assert b"fixed scratch" in msg


def test_static_scratch_no_query_rows_is_a_no_op():
    """No query rows: the other arguments are checked, nothing is launched,
    and the NULL buffers of zero-size tensors are accepted."""
    from sequence_attention_gb300 import _lib
    st, _ = _call_host_only(1, 24, 128, [0, 0], [4608, 4608])
    assert st == _lib.DIT_OK
    st, msg = _call_host_only(1, 24, 96, [0, 0], [4608, 4608])     # an unsupported head dim is still refused
    assert st == _lib.DIT_ERR_UNSUPPORTED, msg
