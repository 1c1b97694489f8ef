"""Failure detection without a GPU fault.

The checked exchange copies a sender's blocks only after the sender has
published the expected epoch on its arrival counter (SGLang Diffusion "The
Ulysses transport": GPU-side sequence counters and a timeout backstop).  The
fault is made on the host: one virtual rank's counter is never advanced, as a
rank that died or a message that was dropped.  The bounded device wait must
run out, report DIT_ERR_TIMEOUT in the status word, leave that rank's blocks
unwritten, and leave the device usable for the next call.
"""
import time

import numpy as np
import pytest
import torch

import synth
from oracle import layout as olayout
from oracle import ulysses as ou
from tests.helpers import bits

pytestmark = pytest.mark.gpu

CASE = (1, 64, 5, 8, 2, 2)        # B, S, H, D, U, R: 4 virtual ranks, padded heads


def _setup():
    import sequence_attention_gb300 as sa
    L = sa.dit_sp_layout_init(*CASE)
    B, S, H, D, U, R = CASE
    planes = [synth.normal((B, S, H, D), 60 + p, 1.0, "bf16").cuda() for p in range(3)]
    send = torch.empty(L.wire_elems(3), dtype=torch.bfloat16, device="cuda")
    sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, planes, send)
    arrival = torch.zeros(U * R, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    return sa, L, planes, send, arrival, status


def test_checked_exchange_equals_plain_when_every_rank_arrived():
    sa, L, planes, send, arrival, status = _setup()
    recv = torch.full_like(send, float("nan"))
    sa.dit_sp_signal(L, arrival, 1)
    sa.dit_a2a_sim_checked(L, sa.DIT_SEQ_TO_HEAD, 3, send, recv, arrival, 1, 50_000_000, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = ou.a2a(olayout.make_layout(*CASE), "s2h", 3, bits(send))
    np.testing.assert_array_equal(bits(recv), ref)


def test_missing_sender_times_out_and_device_stays_usable():
    sa, L, planes, send, arrival, status = _setup()
    U, R = CASE[4], CASE[5]
    dead = 1                                   # rank (r=0, u=1) never publishes epoch 2
    sa.dit_sp_signal(L, arrival, 2, ranks=[i for i in range(U * R) if i != dead])
    recv = torch.full_like(send, float("nan"))
    t0 = time.perf_counter()
    sa.dit_a2a_sim_checked(L, sa.DIT_SEQ_TO_HEAD, 3, send, recv, arrival, 2, 2_000_000, status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == 4             # DIT_ERR_TIMEOUT
    assert elapsed < 5.0                       # bounded: the kernel returned by itself
    # the dead sender's blocks were not written
    ref_layout = olayout.make_layout(*CASE)
    _, recv_base, _ = olayout.buffer_bases(ref_layout, "s2h", 3)
    got = recv.float().cpu().numpy()
    for v in range(U):
        dst = ref_layout.rank(0, v)
        _, _, rc, rd = olayout.a2a_counts(ref_layout, "s2h", 3, dst)
        a = recv_base[dst] + rd[dead % U]
        assert np.isnan(got[a:a + rc[dead % U]]).all()
    # the device is still usable: the same exchange succeeds once the rank arrives
    status.zero_()
    sa.dit_sp_signal(L, arrival, 3)
    recv2 = torch.empty_like(send)
    sa.dit_a2a_sim_checked(L, sa.DIT_SEQ_TO_HEAD, 3, send, recv2, arrival, 3, 50_000_000, status)
    q = synth.normal((1, 128, 2, 64), 1, 0.5, "bf16").cuda()
    o = torch.empty_like(q)
    sa.dit_attention(q, q, q.to(torch.float16), o)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_array_equal(bits(recv2), ou.a2a(ref_layout, "s2h", 3, bits(send)))
    assert torch.isfinite(o.float()).all()


def test_sequence_comparison_wraps():
    sa, L, planes, send, arrival, status = _setup()
    arrival.fill_(-2)                          # 0xFFFFFFFE
    recv = torch.empty_like(send)
    sa.dit_sp_signal(L, arrival, 1)            # the counter wraps to 1 > 0xFFFFFFFE
    sa.dit_a2a_sim_checked(L, sa.DIT_SEQ_TO_HEAD, 3, send, recv, arrival, 1, 50_000_000, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
