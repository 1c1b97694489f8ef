"""A plain C99 program drives the device calls of the ABI: it includes only
include/ditsp.h (and the CUDA runtime for cudaMalloc/cudaMemcpy), runs one
sequence-parallel attention step -- seq->head pack, exchange, unpack (V to
f16), every ring partial in one attention call, the log-sum-exp merge,
head->seq pack, exchange, unpack -- and a CFG combine on device buffers, and
writes the results to files.  No Python touches the device work; the test
compares the files with the fp64 oracle at the parity bars."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import cfg as ocfg
from oracle.numeric import to_f64
from tests.helpers import assert_bf16_close, bits

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
LIBDIR = os.path.join(ROOT, "sequence_attention_gb300")
SRC = os.path.join(ROOT, "tests", "c", "usp_step.c")


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "include", "cuda_runtime.h")):
            return c
    pytest.skip("CUDA runtime headers not found")


@pytest.mark.parametrize("S,H,D,U,R", [(700, 5, 128, 2, 2), (1000, 6, 64, 3, 1)])
def test_c_program_runs_a_step_on_the_device(tmp_path, S, H, D, U, R):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    cuda = _cuda_home()
    exe = tmp_path / "usp_step"
    libdirs = [os.path.join(cuda, d) for d in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib")
               if os.path.exists(os.path.join(cuda, d))]
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Werror", f"-I{INC}", f"-I{os.path.join(cuda, 'include')}", SRC,
           f"-L{LIBDIR}", "-lditsp", f"-Wl,-rpath,{LIBDIR}"]
    for d in libdirs:
        cmd += [f"-L{d}", f"-Wl,-rpath,{d}"]
    cmd += ["-lcudart", "-lm", "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True)
    q = synth.normal((1, S, H, D), 70, 0.5, "bf16")
    k = synth.normal((1, S, H, D), 71, 0.5, "bf16")
    v = synth.normal((1, S, H, D), 72, 0.5, "bf16")
    pred = torch.stack([synth.normal((S * H * D,), 73, 1.0, "bf16"), synth.normal((S * H * D,), 74, 1.0, "bf16")])
    for name, t in (("q", q), ("k", k), ("v", v), ("pred", pred)):
        bits(t).tofile(tmp_path / f"{name}.bin")
    run = subprocess.run([str(exe), str(tmp_path), str(S), str(H), str(D), str(U), str(R)], capture_output=True,
                         text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip() == "ok status=0", run.stdout
    out = np.fromfile(tmp_path / "out.bin", dtype=np.uint16).reshape(1, S, H, D)
    got = to_f64(out, "bf16")
    ref, _ = oatt.attention(to_f64(bits(q), "bf16"), to_f64(bits(k), "bf16"), to_f64(bits(v), "bf16"))
    assert_bf16_close(got, ref, "C program step")
    cfg = to_f64(np.fromfile(tmp_path / "cfg.bin", dtype=np.uint16), "bf16")
    pb = bits(pred)
    want = to_f64(ocfg.cfg_combine_bits(pb, "bf16", 3.5, "bf16"), "bf16")
    u64, c64 = to_f64(pb[0], "bf16"), to_f64(pb[1], "bf16")
    mag = np.abs(want)
    ulp = np.exp2(np.floor(np.log2(np.where(mag > 0, mag, 1.0))) - 7)
    assert np.all(np.abs(cfg - want) <= 3.5 * np.abs(c64 - u64) * 2.0 ** -24 + ulp)
