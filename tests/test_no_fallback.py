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
