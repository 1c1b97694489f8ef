"""The product path has no fallback: without libditsp.so every call raises,
and nothing in the package imports the oracle or computes on the CPU."""
import ast
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sequence_attention_gb300")


def test_missing_library_raises(monkeypatch):
    import sequence_attention_gb300 as sa
    from sequence_attention_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libditsp.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError, match="build"):
        _lib.lib()
    with pytest.raises(ImportError):
        sa.dit_sp_layout_init(1, 64, 4, 64, 2, 1)


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield (node.module or "")


def test_package_never_imports_the_oracle_or_numpy():
    files = [os.path.join(dp, f) for dp, _, fs in os.walk(PKG) for f in fs if f.endswith(".py")]
    assert files
    for f in files:
        if os.path.basename(f) == "build.py":
            continue
        for name in _imports(f):
            root = name.split(".")[0]
            assert root not in ("oracle", "numpy", "scipy", "synth"), f"{f} imports {name}"


def test_host_tensors_are_refused_before_any_launch():
    """A CPU tensor handed to a call would put a host pointer in a kernel;
    the binding refuses it instead (no GPU needed to check)."""
    import torch
    import sequence_attention_gb300 as sa
    L = sa.dit_sp_layout_init(1, 64, 4, 64, 2, 1)
    q = torch.zeros((1, 64, 4, 64), dtype=torch.bfloat16)
    send = torch.zeros(L.wire_elems(3), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, [q, q, q], send)
    o = torch.zeros_like(q)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sa.dit_attention(q, q, q, o)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sa.dit_cfg_combine(torch.zeros((2, 8)), torch.zeros(8), 1.0)
