"""The seeded inputs are reproducible: the same workload draws the same
bytes every time (the bench records their digest in its config), and the
five tensors of a workload come from distinct streams."""
import synth


def test_workload_inputs_are_reproducible():
    w = synth.WORKLOADS["tiny"]
    a = synth.digest(*w.qkv(), w.cfg_pair())
    b = synth.digest(*w.qkv(), w.cfg_pair())
    assert a == b and len(a) == 16


def test_streams_are_distinct():
    w = synth.WORKLOADS["tiny"]
    q, k, v = w.qkv()
    assert len({synth.digest(q), synth.digest(k), synth.digest(v)}) == 3
    assert synth.digest(synth.normal((4, 8), 1)) != synth.digest(synth.normal((4, 8), 2))


def test_digest_sees_every_byte():
    x = synth.normal((3, 5), 7, 1.0, "bf16")
    y = x.clone()
    y.view(-1)[-1] = -y.view(-1)[-1]
    assert synth.digest(x) != synth.digest(y)
