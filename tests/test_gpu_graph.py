"""The whole step captured in a CUDA graph: replaying it gives the same bits
as running it eagerly (every call is a stream-ordered kernel launch and the
plan allocates nothing after it is built)."""
import numpy as np
import pytest
import torch

import synth
from tests.helpers import bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("U,R,fp8", [(4, 1, False), (2, 2, True)])
def test_step_replays_from_a_cuda_graph(U, R, fp8):
    import sequence_attention_gb300 as sa
    from sequence_attention_gb300.usp import UspPlan
    B, S, H, D = 1, 700, 5, 128
    q, k, v = (synth.normal((B, S, H, D), 700 + i, 0.5, "bf16").cuda() for i in range(3))
    pred = torch.stack([synth.normal((S, H * D), 703 + i, 1.0, "bf16") for i in range(2)]).cuda()
    plan = UspPlan(B, S, H, D, U, R, fp8_qv=fp8, fp8_o=fp8)
    eager = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    cfg_eager = torch.empty((S, H * D), dtype=torch.bfloat16, device="cuda")
    plan.run(q, k, v, eager)
    sa.dit_cfg_combine(pred, cfg_eager, 3.5)
    torch.cuda.synchronize()

    out = torch.full_like(eager, float("nan"))
    cfg = torch.full_like(cfg_eager, float("nan"))
    g = plan.capture(q, k, v, out, extra=lambda: sa.dit_cfg_combine(pred, cfg, 3.5))
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(out), bits(eager))
    np.testing.assert_array_equal(bits(cfg), bits(cfg_eager))
    assert int(plan.status.item()) == 0
