"""Every C entry point of libditsp opens an NVTX range named after the call
and closes it on return (tracing for profiler timelines).  Checked on the
CPU through NVTX's own tool-loading hook: a small injection library
(tests/nvtx/record_ranges.c) records the pushes and pops of a child process
that makes calls which finish on the host (layout set-up, argument errors)."""
import os
import shutil
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"


@pytest.fixture(scope="module")
def injection(tmp_path_factory):
    gcc = shutil.which("gcc")
    if not gcc or not os.path.exists(os.path.join(CUDA_INC, "nvtx3", "nvToolsExt.h")):
        pytest.skip("gcc or the NVTX headers are missing")
    lib = tmp_path_factory.mktemp("nvtx") / "librecord_ranges.so"
    subprocess.check_call([gcc, "-shared", "-fPIC", "-O1", f"-I{CUDA_INC}", "-o", str(lib),
                           os.path.join(ROOT, "tests", "nvtx", "record_ranges.c")])
    return str(lib)


def test_entry_points_open_and_close_named_ranges(injection, tmp_path):
    log = tmp_path / "ranges.log"
    code = textwrap.dedent("""
        import ctypes, sys
        sys.path.insert(0, %r)
        from sequence_attention_gb300 import _lib as dl
        L = dl.lib()
        lay = dl.DitSpLayout()
        assert L.dit_sp_layout_init(1, 64, 4, 64, 2, 1, ctypes.byref(lay)) == 0
        assert L.dit_sp_layout_init_ex(1, 64, 4, 64, 2, 1, 99, ctypes.byref(lay)) != 0      # unknown flag bits
        c = (ctypes.c_int64 * 2)()
        assert L.dit_sp_a2a_counts(ctypes.byref(lay), 0, 3, 0, c, c, c, c) == 0
        assert L.dit_cfg_combine(None, 1, 8, 1.0, None, 1, None) != 0                      # NULL buffers
        assert L.dit_ulysses_pack(None, 0, 3, None, 1, None, 1, None) != 0                 # NULL layout
    """ % ROOT)
    env = dict(os.environ, NVTX_INJECTION64_PATH=injection, DITSP_NVTX_LOG=str(log))
    subprocess.run([sys.executable, "-c", code], env=env, check=True, timeout=300)
    lines = log.read_text().splitlines()
    pushes = [ln.split(" ", 1)[1] for ln in lines if ln.startswith("push ")]
    assert pushes == ["dit_sp_layout_init", "dit_sp_layout_init_ex", "dit_sp_layout_init_ex",
                      "dit_sp_a2a_counts", "dit_cfg_combine", "dit_ulysses_pack"], lines
    depth = 0
    for ln in lines:                          # every push closed, never below zero
        depth += 1 if ln.startswith("push ") else -1
        assert depth >= 0, lines
    assert depth == 0, lines


def test_every_exported_call_has_a_range():
    """The sources put a range at the top of every exported call except the
    two that only return strings."""
    import re
    from sequence_attention_gb300._lib import EXPORTS
    csrc = os.path.join(ROOT, "sequence_attention_gb300", "csrc")
    text = "".join(open(os.path.join(csrc, f)).read() for f in os.listdir(csrc) if f.endswith(".cu"))
    for name in EXPORTS:
        if name in ("dit_status_string", "dit_last_error"):
            continue
        m = re.search(r'extern "C" [^\n]*\b%s\([^{]*\{\n\s*NvtxRange nvtx_range\("%s"\);' % (name, name), text)
        assert m, name
