"""The boundary is a plain C ABI: a C99 program that includes only
include/ditsp.h compiles with gcc, links against libditsp.so and runs the
host-side calls (layout, all-to-all counts, argument validation, error
strings, the empty exchange) without Python, torch or a GPU; and the last-error string is kept
per calling thread."""
import ctypes
import os
import shutil
import subprocess
import threading

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
LIBDIR = os.path.join(ROOT, "sequence_attention_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "ditsp.h"

int main(void) {
    dit_sp_layout L;
    int64_t sc[5], sd[5], rc[5], rd[5];
    dit_status s = dit_sp_layout_init(2, 7145, 24, 128, 5, 2, &L);
    if (s != DIT_OK) { printf("init %d %s\n", (int)s, dit_last_error()); return 1; }
    printf("Hp=%d Hl=%d S_cap=%d ring=%d,%d\n", L.Hp, L.Hl, L.S_cap, L.ring_len[0], L.ring_len[1]);
    s = dit_sp_a2a_counts(&L, DIT_SEQ_TO_HEAD, 3, 0, sc, sd, rc, rd);
    if (s != DIT_OK) return 2;
    printf("send0=%lld recv4=%lld\n", (long long)sc[0], (long long)rc[4]);
    s = dit_sp_layout_init_ex(1, 4481, 24, 128, 4, 2, DIT_LAYOUT_PAD_LCM64 | DIT_LAYOUT_NOPAD_HEADS, &L);
    printf("S_pad=%d Hp=%d head_len0=%d\n", L.S_pad, L.Hp, L.head_len[0]);
    s = dit_sp_layout_init(0, 8, 1, 8, 1, 1, &L);        /* B = 0 is refused */
    printf("bad=%s msg=%s\n", dit_status_string(s), strlen(dit_last_error()) > 0 ? "yes" : "no");
    /* an empty sequence: the exchange moves nothing and takes NULL buffers */
    s = dit_sp_layout_init(1, 0, 4, 64, 2, 2, &L);
    const void* none[3] = {NULL, NULL, NULL};
    dit_status e1 = dit_ulysses_pack(&L, DIT_SEQ_TO_HEAD, 3, none, DIT_BF16, NULL, DIT_BF16, NULL);
    dit_status e2 = dit_a2a_sim(&L, DIT_SEQ_TO_HEAD, 3, NULL, NULL, DIT_BF16, NULL);
    printf("empty=%s,%s,%s\n", dit_status_string(s), dit_status_string(e1), dit_status_string(e2));
    return 0;
}
"""


@pytest.fixture(scope="module")
def built():
    lib = os.path.join(LIBDIR, "libditsp.so")
    if not os.path.exists(lib):
        pytest.skip("libditsp.so not built")
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    return lib


def test_plain_c_program_uses_the_library(built, tmp_path):
    src = tmp_path / "use_ditsp.c"
    exe = tmp_path / "use_ditsp"
    src.write_text(PROGRAM)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", f"-I{INC}", str(src), f"-L{LIBDIR}", "-lditsp",
                    f"-Wl,-rpath,{LIBDIR}", "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    assert out[0] == "Hp=25 Hl=5 S_cap=3573 ring=3573,3572"
    # rank 0 sends each peer its 715 rows of 5 heads, 3 planes, B = 2
    assert out[1] == f"send0={3 * 2 * 715 * 5 * 128} recv4={3 * 2 * 714 * 5 * 128}"
    assert out[2] == "S_pad=4544 Hp=24 head_len0=6"
    assert out[3] == "bad=DIT_ERR_INVALID_ARG msg=yes"
    assert out[4] == "empty=DIT_OK,DIT_OK,DIT_OK"


def test_last_error_is_per_thread():
    from sequence_attention_gb300 import _lib
    L = _lib.lib()
    msgs = {}

    def worker(i):
        lay = _lib.DitSpLayout()
        # a different invalid Ulysses degree on every thread
        for _ in range(200):
            assert L.dit_sp_layout_init(1, 8, 1, 8, 100 + i, 1, ctypes.byref(lay)) == _lib.DIT_ERR_INVALID_ARG
            msgs.setdefault(i, set()).add(L.dit_last_error().decode())

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    for i in range(8):
        assert len(msgs[i]) == 1 and f"U={100 + i}" in next(iter(msgs[i])), msgs[i]
