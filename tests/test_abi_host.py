"""The C ABI on the host: the library loads, exports every symbol the header
declares, its layout bookkeeping equals the oracle's, and bad arguments are
rejected before anything is launched (these calls never reach a GPU)."""
import ctypes
import os
import re

import pytest

from oracle import layout as olayout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ditsp.h")


@pytest.fixture(scope="module")
def dl():
    if not os.path.exists(os.path.join(ROOT, "sequence_attention_gb300", "libditsp.so")):
        import __graft_entry__
        __graft_entry__.build()
    from sequence_attention_gb300 import _lib
    return _lib


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DIT_API\s+[\w\s\*]*?\b(dit_\w+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("dit_attn_partial", "dit_attn_merge_lse", "dit_ulysses_pack", "dit_ulysses_unpack",
              "dit_a2a_sim", "dit_cfg_combine", "dit_attention", "dit_sp_layout_init"):
        assert n in names


def test_library_exports_every_declared_symbol(dl):
    raw = ctypes.CDLL(dl.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name
    assert set(declared_functions()) == set(dl.EXPORTS)


def test_binding_imports(dl):
    import sequence_attention_gb300 as sa
    assert os.path.samefile(sa.library_path(), dl.LIB_PATH)


@pytest.mark.parametrize("dims", [(1, 256, 4, 64, 2, 2), (1, 4608, 24, 128, 4, 1), (1, 4481, 24, 128, 4, 2),
                                  (2, 7145, 24, 128, 5, 2), (1, 75600, 40, 128, 8, 4), (1, 3, 2, 8, 2, 2),
                                  (1, 0, 1, 8, 3, 2), (3, 17, 5, 8, 64, 1)])
def test_layout_init_matches_oracle(dl, dims):
    import sequence_attention_gb300 as sa
    L = sa.dit_sp_layout_init(*dims)
    ref = olayout.make_layout(*dims)
    assert (L.Hp, L.Hl, L.S_cap) == (ref.Hp, ref.Hl, ref.S_cap)
    assert L.ring_len == list(ref.ring_len) and L.ring_off == list(ref.ring_off)
    assert L.rank_len == list(ref.rank_len) and L.rank_off == list(ref.rank_off)
    assert L.ring_real == [ref.real_rows(r) for r in range(ref.R)]


@pytest.mark.parametrize("flags", [(False, False), (True, True), (False, True)])
@pytest.mark.parametrize("dims", [(1, 4481, 24, 128, 4, 2), (2, 7145, 24, 128, 5, 2), (1, 75600, 40, 128, 8, 4),
                                  (1, 3, 2, 8, 2, 2), (1, 0, 1, 8, 3, 2), (3, 17, 5, 8, 64, 1)])
def test_layout_modes_match_oracle(dl, dims, flags):
    import sequence_attention_gb300 as sa
    L = sa.dit_sp_layout_init(*dims, pad_heads=flags[0], pad_lcm64=flags[1])
    ref = olayout.make_layout(*dims, pad_heads=flags[0], pad_lcm64=flags[1])
    assert (L.Hp, L.Hl, L.S_cap, L.S_pad, L.S) == (ref.Hp, ref.Hl, ref.S_cap, ref.S_pad, ref.S)
    assert L.head_len == list(ref.head_len) and L.head_off == list(ref.head_off)
    assert L.ring_len == list(ref.ring_len) and L.ring_off == list(ref.ring_off)
    assert L.rank_len == list(ref.rank_len) and L.rank_off == list(ref.rank_off)
    assert L.ring_real == [ref.real_rows(r) for r in range(ref.R)]
    for d, name in ((0, "s2h"), (1, "h2s")):
        for rank in range(min(dims[4] * dims[5], 9)):
            got = sa.dit_sp_a2a_counts(L, d, 3 if d == 0 else 1, rank)
            exp = olayout.a2a_counts(ref, name, 3 if d == 0 else 1, rank)
            assert [list(x) for x in got] == [list(x) for x in exp]


def test_layout_init_rejects_unknown_flags(dl):
    lay = dl.DitSpLayout()
    assert dl.lib().dit_sp_layout_init_ex(1, 8, 2, 8, 2, 1, 4, ctypes.byref(lay)) == dl.DIT_ERR_INVALID_ARG


@pytest.mark.parametrize("direction,np_", [(0, 3), (1, 1), (0, 1)])
def test_a2a_counts_match_oracle(dl, direction, np_):
    import sequence_attention_gb300 as sa
    dims = (2, 7145, 24, 128, 5, 2)
    L = sa.dit_sp_layout_init(*dims)
    ref = olayout.make_layout(*dims)
    for rank in range(10):
        got = sa.dit_sp_a2a_counts(L, direction, np_, rank)
        exp = olayout.a2a_counts(ref, "s2h" if direction == 0 else "h2s", np_, rank)
        assert [list(x) for x in got] == [list(x) for x in exp]


@pytest.mark.parametrize("args", [(0, 8, 1, 8, 1, 1), (1, -1, 1, 8, 1, 1), (1, 8, 1, 8, 65, 1),
                                  (1, 8, 1, 8, 1, 9), (1, 8, 1, 8, 16, 8)])
def test_layout_init_rejects_bad_sizes(dl, args):
    import sequence_attention_gb300 as sa
    with pytest.raises(sa.DitError) as e:
        sa.dit_sp_layout_init(*args)
    assert e.value.status == dl.DIT_ERR_INVALID_ARG


def test_validation_happens_before_any_launch(dl):
    """Each call below fails validation; none of them touches the CUDA runtime,
    so they behave the same with or without a GPU."""
    L = dl.lib()
    lay = dl.DitSpLayout()
    assert L.dit_sp_layout_init(1, 64, 4, 64, 2, 2, ctypes.byref(lay)) == 0
    bad = dl.DitSpLayout.from_buffer_copy(lay)
    bad.rank_len[0] += 1                      # corrupted table
    ptrs = (ctypes.c_void_p * 3)(16, 32, 48)
    st = L.dit_ulysses_pack(ctypes.byref(bad), 0, 3, ptrs, dl.DIT_BF16, ctypes.c_void_p(64), dl.DIT_BF16, None)
    assert st == dl.DIT_ERR_INVALID_ARG and b"inconsistent" in L.dit_last_error()
    # misaligned send buffer
    st = L.dit_ulysses_pack(ctypes.byref(lay), 0, 3, ptrs, dl.DIT_BF16, ctypes.c_void_p(8), dl.DIT_BF16, None)
    assert st == dl.DIT_ERR_INVALID_ARG
    # head-to-seq with 3 planes
    st = L.dit_ulysses_pack(ctypes.byref(lay), 1, 3, ptrs, dl.DIT_BF16, ctypes.c_void_p(64), dl.DIT_BF16, None)
    assert st == dl.DIT_ERR_INVALID_ARG
    # a2a with identical send/recv
    st = L.dit_a2a_sim(ctypes.byref(lay), 0, 3, ctypes.c_void_p(64), ctypes.c_void_p(64), dl.DIT_BF16, None)
    assert st == dl.DIT_ERR_INVALID_ARG
    # cfg: N < 0, NULL, overlap
    assert L.dit_cfg_combine(ctypes.c_void_p(64), dl.DIT_BF16, -1, 1.0, ctypes.c_void_p(128), dl.DIT_BF16, None) \
        == dl.DIT_ERR_INVALID_ARG
    assert L.dit_cfg_combine(None, dl.DIT_BF16, 8, 1.0, ctypes.c_void_p(128), dl.DIT_BF16, None) \
        == dl.DIT_ERR_INVALID_ARG
    assert L.dit_cfg_combine(ctypes.c_void_p(64), dl.DIT_BF16, 64, 1.0, ctypes.c_void_p(96), dl.DIT_BF16, None) \
        == dl.DIT_ERR_INVALID_ARG
    assert L.dit_cfg_combine(ctypes.c_void_p(64), 7, 8, 1.0, ctypes.c_void_p(4096), dl.DIT_BF16, None) \
        == dl.DIT_ERR_INVALID_ARG
    assert L.dit_cfg_combine(ctypes.c_void_p(64), dl.DIT_BF16, 0, 1.0, ctypes.c_void_p(4096), dl.DIT_BF16, None) \
        == dl.DIT_OK                           # empty: nothing to do


def test_checked_exchange_argument_checks(dl):
    L = dl.lib()
    lay = dl.DitSpLayout()
    assert L.dit_sp_layout_init(1, 64, 4, 64, 2, 2, ctypes.byref(lay)) == 0
    send, recv, arr = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), ctypes.c_void_p(3 << 20)
    assert L.dit_a2a_sim_checked(ctypes.byref(lay), 0, 3, send, recv, dl.DIT_BF16, arr, 1, 0, None, None) \
        == dl.DIT_ERR_INVALID_ARG                            # timeout must be positive
    assert L.dit_a2a_sim_checked(ctypes.byref(lay), 0, 3, send, recv, dl.DIT_BF16, arr, 1, 20_000_000_000, None,
                                 None) == dl.DIT_ERR_INVALID_ARG   # and at most 10 s
    assert L.dit_a2a_sim_checked(ctypes.byref(lay), 0, 3, send, recv, dl.DIT_BF16, None, 1, 1000, None, None) \
        == dl.DIT_ERR_INVALID_ARG                            # counters required
    assert L.dit_sp_signal(ctypes.byref(lay), ctypes.c_void_p(2), None, 1, None) == dl.DIT_ERR_INVALID_ARG


def _view(ptr, sb=0, ss=0, sh=0):
    from sequence_attention_gb300._lib import DitView
    v = DitView()
    v.ptr, v.stride_b, v.stride_s, v.stride_h = ptr, sb, ss, sh
    return v


def test_attention_argument_checks(dl):
    from sequence_attention_gb300._lib import DitLseView
    L = dl.lib()
    q = _view(1 << 20, 64 * 4 * 128, 4 * 128, 128)
    lse = DitLseView()
    ok = dict(B=1, H=4, D=128, Sq=64, Sk=64)

    def call(**kw):
        a = dict(ok, qk=dl.DIT_BF16, v=dl.DIT_F16, o=dl.DIT_BF16, q=q)
        a.update(kw)
        return L.dit_attention(a["B"], a["H"], a["D"], 0.1, a["Sq"], a["Sk"], a["q"], a["qk"], q, q,
                               a["v"], q, a["o"], lse, None, None)

    assert call(D=96) == dl.DIT_ERR_UNSUPPORTED          # tensor-core path: D in {64, 128}
    assert call(qk=dl.DIT_F32) == dl.DIT_ERR_UNSUPPORTED  # fp32 Q/K need fp32 V and O
    assert call(v=dl.DIT_F32) == dl.DIT_ERR_UNSUPPORTED
    assert call(B=0) == dl.DIT_ERR_INVALID_ARG
    assert call(Sq=-1) == dl.DIT_ERR_INVALID_ARG
    assert call(q=_view(1 << 20, 64 * 4 * 128, 4 * 128 + 1, 128)) == dl.DIT_ERR_INVALID_ARG  # odd stride
    assert call(q=_view((1 << 20) + 8, 64 * 4 * 128, 4 * 128, 128)) == dl.DIT_ERR_INVALID_ARG  # misaligned
    assert call(q=_view(0)) == dl.DIT_ERR_INVALID_ARG    # NULL
    lens = (ctypes.c_int * 9)(*([8] * 9))
    st = L.dit_attn_partial(1, 4, 128, 0.1, 9, lens, 1, lens, q, dl.DIT_BF16, q, q, dl.DIT_F16, q,
                            dl.DIT_BF16, lse, None, None)
    assert st == dl.DIT_ERR_INVALID_ARG                  # more than 8 query blocks


def test_attention_output_aliasing_is_refused(dl):
    """A zero output stride on a dimension with more than one index would
    send two results to one address; it is refused before any launch (a
    zero stride on a dimension of one index is fine)."""
    from sequence_attention_gb300._lib import DitLseView
    L = dl.lib()
    q = _view(1 << 20, 64 * 4 * 128, 4 * 128, 128)
    lse = DitLseView()

    def attention(o, B=1, Sq=64):
        return L.dit_attention(B, 4, 128, 0.1, Sq, 64, q, dl.DIT_BF16, q, q, dl.DIT_F16, o, dl.DIT_BF16, lse,
                               None, None)

    assert attention(_view(1 << 20, 64 * 4 * 128, 0, 128)) == dl.DIT_ERR_INVALID_ARG      # rows alias
    assert attention(_view(1 << 20, 64 * 4 * 128, 4 * 128, 0)) == dl.DIT_ERR_INVALID_ARG  # heads alias
    assert attention(_view(1 << 20, 0, 4 * 128, 128), B=2) == dl.DIT_ERR_INVALID_ARG       # batches alias
    # one query row: a zero row stride is fine, the call goes on to the device
    assert attention(_view(1 << 20, 64 * 4 * 128, 0, 128), Sq=1) != dl.DIT_ERR_INVALID_ARG
    lens = (ctypes.c_int * 2)(64, 64)
    o = _view(1 << 20, 64 * 4 * 128, 4 * 128, 128)
    o.stride_q, o.stride_kv = 0, 2 * 64 * 4 * 128
    st = L.dit_attn_partial(1, 4, 128, 0.1, 2, lens, 2, lens, q, dl.DIT_BF16, q, q, dl.DIT_F16, o,
                            dl.DIT_BF16, lse, None, None)
    assert st == dl.DIT_ERR_INVALID_ARG                  # query blocks alias
    o.stride_q, o.stride_kv = 2 * 64 * 4 * 128, 0
    st = L.dit_attn_partial(1, 4, 128, 0.1, 2, lens, 2, lens, q, dl.DIT_BF16, q, q, dl.DIT_F16, o,
                            dl.DIT_BF16, lse, None, None)
    assert st == dl.DIT_ERR_INVALID_ARG                  # key blocks alias


def test_status_strings(dl):
    L = dl.lib()
    assert L.dit_status_string(0) == b"DIT_OK"
    assert L.dit_status_string(4) == b"DIT_ERR_TIMEOUT"
    assert L.dit_status_string(99) == b"DIT_ERR_UNKNOWN"


def test_new_entry_points_validate_before_any_launch(dl):
    """Argument errors of the receive-preparation, paired-stream, e4m3 and
    varlen calls are reported before anything touches the CUDA runtime."""
    L = dl.lib()
    lay = dl.DitSpLayout()
    assert L.dit_sp_layout_init(1, 64, 4, 64, 2, 1, ctypes.byref(lay)) == 0
    p = (ctypes.c_void_p * 3)(1 << 20, 2 << 20, 3 << 20)
    dts = (ctypes.c_int * 3)(dl.DIT_BF16, dl.DIT_BF16, dl.DIT_F16)
    buf = ctypes.c_void_p(4 << 20)
    tab = ctypes.c_void_p(5 << 20)
    # RoPE on a plane the call does not have
    assert L.dit_ulysses_unpack_rope(ctypes.byref(lay), 1, buf, dl.DIT_BF16, p, dts, tab, tab, 0b10, None,
                                     None) == dl.DIT_ERR_INVALID_ARG
    # RoPE without tables
    assert L.dit_ulysses_unpack_rope(ctypes.byref(lay), 2, buf, dl.DIT_BF16, p, dts, None, None, 0b1, None,
                                     None) == dl.DIT_ERR_INVALID_ARG
    # more text rows than the sequence has
    assert L.dit_ulysses_pack_joint(ctypes.byref(lay), 3, p, p, 65, dl.DIT_BF16, buf, dl.DIT_BF16,
                                    None) == dl.DIT_ERR_INVALID_ARG
    # image stream missing while S_txt < S
    assert L.dit_ulysses_pack_joint(ctypes.byref(lay), 3, p, None, 10, dl.DIT_BF16, buf, dl.DIT_BF16,
                                    None) == dl.DIT_ERR_INVALID_ARG
    # e4m3 is a wire type only, and its head dim must be a power of two in [16, 256]
    assert L.dit_ulysses_pack(ctypes.byref(lay), 0, 3, p, dl.DIT_E4M3, buf, dl.DIT_BF16,
                              None) == dl.DIT_ERR_INVALID_ARG
    lay24 = dl.DitSpLayout()
    assert L.dit_sp_layout_init(1, 64, 4, 24, 2, 1, ctypes.byref(lay24)) == 0
    assert L.dit_ulysses_pack(ctypes.byref(lay24), 0, 3, p, dl.DIT_BF16, buf, dl.DIT_E4M3,
                              None) == dl.DIT_ERR_UNSUPPORTED
    assert L.dit_a2a_sim(ctypes.byref(lay24), 0, 3, buf, ctypes.c_void_p(6 << 20), dl.DIT_E4M3,
                         None) == dl.DIT_ERR_UNSUPPORTED
    # varlen: offsets must not decrease
    v = dl.DitView()
    v.ptr = 7 << 20
    v.stride_s, v.stride_h = 128, 64
    cu_q = (ctypes.c_int * 3)(0, 5, 4)
    cu_k = (ctypes.c_int * 3)(0, 5, 10)
    assert L.dit_attn_varlen(2, 64, 0.125, 2, cu_q, cu_k, v, dl.DIT_BF16, v, v, dl.DIT_F16, v, dl.DIT_BF16,
                             dl.DitLseView(), None, None) == dl.DIT_ERR_INVALID_ARG
    assert L.dit_attn_varlen(2, 64, 0.125, 0, None, None, v, dl.DIT_BF16, v, v, dl.DIT_F16, v, dl.DIT_BF16,
                             dl.DitLseView(), None, None) == dl.DIT_OK          # nothing to do


def test_one_pass_permutation_validates_before_any_launch(dl):
    """dit_ulysses_seq_to_head / dit_ulysses_head_to_seq refuse bad arguments
    on the host: no launch, no CUDA call."""
    L = dl.lib()
    lay = dl.DitSpLayout()
    assert L.dit_sp_layout_init(1, 64, 4, 64, 2, 1, ctypes.byref(lay)) == 0
    p = (ctypes.c_void_p * 3)(1 << 20, 2 << 20, 3 << 20)
    mis = (ctypes.c_void_p * 3)((1 << 20) + 8, 2 << 20, 3 << 20)
    dts = (ctypes.c_int * 3)(dl.DIT_BF16, dl.DIT_BF16, dl.DIT_F16)
    bad_dts = (ctypes.c_int * 3)(dl.DIT_BF16, dl.DIT_E4M3, dl.DIT_F16)
    tab = ctypes.c_void_p(5 << 20)
    lp = ctypes.byref(lay)
    E = dl.DIT_ERR_INVALID_ARG
    s2h, h2s = L.dit_ulysses_seq_to_head, L.dit_ulysses_head_to_seq
    assert s2h(lp, 0, p, None, 0, dl.DIT_BF16, p, dts, None, None, 0, None, None) == E        # no planes
    assert s2h(lp, 4, p, None, 0, dl.DIT_BF16, p, dts, None, None, 0, None, None) == E        # too many
    assert s2h(lp, 3, p, None, 0, dl.DIT_E4M3, p, dts, None, None, 0, None, None) == E        # no e4m3 source
    assert s2h(lp, 3, p, None, 0, dl.DIT_BF16, p, bad_dts, None, None, 0, None, None) == E    # nor destination
    assert s2h(lp, 3, p, None, 65, dl.DIT_BF16, p, dts, None, None, 0, None, None) == E       # split > S
    assert s2h(lp, 3, p, None, 10, dl.DIT_BF16, p, dts, None, None, 0, None, None) == E       # second stream
    assert s2h(lp, 3, mis, None, 0, dl.DIT_BF16, p, dts, None, None, 0, None, None) == E      # misaligned
    assert s2h(lp, 3, p, None, 0, dl.DIT_BF16, mis, dts, None, None, 0, None, None) == E
    assert s2h(lp, 2, p, None, 0, dl.DIT_BF16, p, dts, None, None, 0b100, None, None) == E    # missing plane
    assert s2h(lp, 3, p, None, 0, dl.DIT_BF16, p, dts, None, None, 0b011, None, None) == E    # no tables
    assert s2h(lp, 3, p, None, 0, dl.DIT_BF16, p, dts, tab, None, 0b011, None, None) == E
    assert s2h(None, 3, p, None, 0, dl.DIT_BF16, p, dts, None, None, 0, None, None) == E      # no layout
    buf = ctypes.c_void_p(4 << 20)
    assert h2s(lp, None, dl.DIT_BF16, buf, None, 0, dl.DIT_BF16, None) == E
    assert h2s(lp, buf, dl.DIT_BF16, None, None, 0, dl.DIT_BF16, None) == E
    assert h2s(lp, buf, dl.DIT_BF16, buf, None, 10, dl.DIT_BF16, None) == E                   # second stream
    assert h2s(lp, buf, dl.DIT_E4M3, buf, None, 0, dl.DIT_BF16, None) == E
    assert h2s(lp, buf, dl.DIT_BF16, buf, None, -1, dl.DIT_BF16, None) == E
    lay24 = dl.DitSpLayout()
    assert L.dit_sp_layout_init(1, 64, 4, 12, 2, 1, ctypes.byref(lay24)) == 0
    assert s2h(ctypes.byref(lay24), 3, p, None, 0, dl.DIT_BF16, p, dts, None, None, 0, None,
               None) == dl.DIT_ERR_UNSUPPORTED                                                 # D % 8 != 0
    lay512 = dl.DitSpLayout()
    assert L.dit_sp_layout_init(1, 64, 2, 512, 2, 1, ctypes.byref(lay512)) == 0
    assert s2h(ctypes.byref(lay512), 3, p, None, 0, dl.DIT_BF16, p, dts, tab, tab, 0b011, None,
               None) == dl.DIT_ERR_UNSUPPORTED                                                 # rotary D > 384
    # a corrupted layout table is refused
    bad = dl.DitSpLayout.from_buffer_copy(lay)
    bad.ring_real[0] = 3
    assert h2s(ctypes.byref(bad), buf, dl.DIT_BF16, buf, None, 0, dl.DIT_BF16, None) == E
    # S = 0 moves nothing, whatever the pointers
    lay0 = dl.DitSpLayout()
    assert L.dit_sp_layout_init(2, 0, 4, 64, 2, 2, ctypes.byref(lay0)) == 0
    null3 = (ctypes.c_void_p * 3)(None, None, None)
    assert s2h(ctypes.byref(lay0), 3, null3, None, 0, dl.DIT_BF16, null3, dts, None, None, 0, None, None) == 0
    assert h2s(ctypes.byref(lay0), None, dl.DIT_BF16, None, None, 0, dl.DIT_BF16, None) == 0


def test_layout_with_lcm_padding_changes_wire_sizes(dl):
    import sequence_attention_gb300 as sa
    L = sa.dit_sp_layout_init(1, 4481, 24, 128, 4, 2, pad_lcm64=True)
    assert L.S_pad == 4544 and L.wire_elems(3) == 3 * 4544 * 24 * 128
    assert L.wire_bytes_e4m3(2) == 2 * 4544 * 24 * 144
    assert [L.real_rows(r) for r in range(2)] == [2272, 2209]


@pytest.mark.parametrize("pad_lcm64", [False, True])
def test_empty_layout_moves_nothing(dl, pad_lcm64):
    """S = 0: every buffer of the exchange is empty (an allocator gives NULL
    for zero bytes), so each call checks its other arguments and returns
    DIT_OK without a launch; the answer to a bad argument does not change."""
    L = dl.lib()
    lay = dl.DitSpLayout()
    flags = dl.DIT_LAYOUT_PAD_LCM64 if pad_lcm64 else 0
    assert L.dit_sp_layout_init_ex(3, 0, 9, 32, 1, 4, flags, ctypes.byref(lay)) == 0
    assert lay.S_pad == 0
    null3 = (ctypes.c_void_p * 3)(None, None, None)
    dts = (ctypes.c_int * 3)(dl.DIT_BF16, dl.DIT_BF16, dl.DIT_F16)
    ok = dl.DIT_OK
    for wire in (dl.DIT_BF16, dl.DIT_E4M3):
        assert L.dit_ulysses_pack(ctypes.byref(lay), 0, 3, null3, dl.DIT_BF16, None, wire, None) == ok
        assert L.dit_ulysses_pack(ctypes.byref(lay), 1, 1, null3, dl.DIT_BF16, None, wire, None) == ok
        assert L.dit_a2a_sim(ctypes.byref(lay), 0, 3, None, None, wire, None) == ok
        assert L.dit_ulysses_unpack(ctypes.byref(lay), 0, 3, None, wire, null3, dts, None, None) == ok
        assert L.dit_ulysses_unpack(ctypes.byref(lay), 1, 1, None, wire, null3, dts, None, None) == ok
        assert L.dit_ulysses_unpack_rope(ctypes.byref(lay), 3, None, wire, null3, dts, None, None, 0b011, None,
                                         None) == ok
        assert L.dit_ulysses_pack_joint(ctypes.byref(lay), 3, None, None, 0, dl.DIT_BF16, None, wire, None) == ok
        assert L.dit_ulysses_unpack_joint(ctypes.byref(lay), None, wire, None, None, 0, dl.DIT_BF16, None) == ok
        assert L.dit_a2a_sim_checked(ctypes.byref(lay), 0, 3, None, None, wire, ctypes.c_void_p(1 << 20), 1,
                                     1000, None, None) == ok
    # the other arguments are still checked
    assert L.dit_ulysses_pack(ctypes.byref(lay), 1, 3, null3, dl.DIT_BF16, None, dl.DIT_BF16, None) \
        == dl.DIT_ERR_INVALID_ARG                            # head-to-seq with 3 planes
    assert L.dit_ulysses_unpack(ctypes.byref(lay), 0, 3, None, dl.DIT_BF16, null3, None, None, None) \
        == dl.DIT_ERR_INVALID_ARG                            # no destination types
    assert L.dit_a2a_sim_checked(ctypes.byref(lay), 0, 3, None, None, dl.DIT_BF16, None, 1, 1000, None, None) \
        == dl.DIT_ERR_INVALID_ARG                            # counters required
    lay24 = dl.DitSpLayout()
    assert L.dit_sp_layout_init(1, 0, 4, 24, 2, 1, ctypes.byref(lay24)) == 0
    assert L.dit_ulysses_pack(ctypes.byref(lay24), 0, 3, null3, dl.DIT_BF16, None, dl.DIT_E4M3, None) \
        == dl.DIT_ERR_UNSUPPORTED                            # e4m3 head dim, as with S > 0


def test_attention_without_rows_touches_nothing(dl):
    """No query rows: attention and the merge check their sizes, types and
    strides, then return DIT_OK without a launch, with NULL buffers."""
    from sequence_attention_gb300._lib import DitLseView
    L = dl.lib()
    null, lse = _view(0, 0, 4 * 128, 128), DitLseView()
    assert L.dit_attention(1, 4, 128, 0.1, 0, 64, null, dl.DIT_BF16, null, null, dl.DIT_F16, null,
                           dl.DIT_BF16, lse, None, None) == dl.DIT_OK
    assert L.dit_attention(1, 4, 96, 0.1, 0, 64, null, dl.DIT_BF16, null, null, dl.DIT_F16, null,
                           dl.DIT_BF16, lse, None, None) == dl.DIT_ERR_UNSUPPORTED    # D still checked
    zeros = (ctypes.c_int * 2)(0, 0)
    lens = (ctypes.c_int * 2)(5, 0)
    o = _view(0, 0, 4 * 128, 128)
    o.stride_q, o.stride_kv = 2 * 8 * 4 * 128, 8 * 4 * 128   # blocks of the (empty) output stay apart
    assert L.dit_attn_partial(1, 4, 128, 0.1, 2, zeros, 2, lens, null, dl.DIT_BF16, null, null, dl.DIT_F16,
                              o, dl.DIT_F32, lse, None, None) == dl.DIT_OK
    assert L.dit_attn_merge_lse(1, 4, 128, 2, zeros, 2, null, dl.DIT_F32, lse, null, dl.DIT_BF16, lse,
                                None) == dl.DIT_OK
    assert L.dit_attn_merge_lse(1, 4, 128, 2, lens, 2, null, dl.DIT_F32, lse, null, dl.DIT_BF16, lse,
                                None) == dl.DIT_ERR_INVALID_ARG                      # rows need buffers
    cu = (ctypes.c_int * 3)(0, 0, 0)
    assert L.dit_attn_varlen(4, 128, 0.1, 2, cu, cu, null, dl.DIT_BF16, null, null, dl.DIT_F16, null,
                             dl.DIT_BF16, lse, None, None) == dl.DIT_OK
    # rows but NULL Q is still an error; NULL K and V with keys too
    assert L.dit_attention(1, 4, 128, 0.1, 8, 0, null, dl.DIT_BF16, null, null, dl.DIT_F16, null,
                           dl.DIT_BF16, lse, None, None) == dl.DIT_ERR_INVALID_ARG
    q = _view(1 << 20, 64 * 4 * 128, 4 * 128, 128)
    assert L.dit_attention(1, 4, 128, 0.1, 8, 8, q, dl.DIT_BF16, null, null, dl.DIT_F16, q,
                           dl.DIT_BF16, lse, None, None) == dl.DIT_ERR_INVALID_ARG


def test_plan_partial_type(dl):
    """Ring partials are f16 when V is f16 and the output 16-bit (a partial
    lies within V's range), f32 otherwise; f16 partials without f16 V are
    refused.  Plans are built on the host here: nothing is launched."""
    import torch
    from sequence_attention_gb300.usp import UspPlan
    rm = {"ring_merge": "partials"}
    assert UspPlan(1, 64, 2, 64, 2, 2, device="cpu", **rm).parts.dtype == torch.float16
    assert UspPlan(1, 64, 2, 64, 2, 2, device="cpu", out_dtype=torch.float32, **rm).parts.dtype == torch.float32
    assert UspPlan(1, 64, 2, 64, 2, 2, device="cpu", v_dtype=torch.bfloat16, **rm).parts.dtype == torch.float32
    assert UspPlan(1, 64, 2, 64, 2, 2, device="cpu", parts_dtype=torch.float32, **rm).parts.dtype == torch.float32
    with pytest.raises(ValueError):
        UspPlan(1, 64, 2, 64, 2, 2, device="cpu", v_dtype=torch.bfloat16, parts_dtype=torch.float16)
    # folding the ring blocks in the attention needs no partial buffers
    fold = UspPlan(1, 64, 2, 64, 2, 2, device="cpu")
    assert fold.ring_merge == "fold" and fold.parts is None and fold.lse_parts is None
    # with the one-pass exchange the folded attention writes the output in place
    assert fold.steps() == ["seq_to_head", "attn_ring"]
    out = torch.empty((1, 64, 2, 64), dtype=torch.bfloat16)
    assert fold.direct_out(out) and not fold.direct_out(out[:, :32])
    assert not UspPlan(1, 64, 2, 64, 2, 2, device="cpu", exchange="a2a").direct_out(out)
    assert UspPlan(1, 64, 2, 64, 2, 2, device="cpu", exchange="a2a").steps()[-1] == "unpack_h2s"
    assert UspPlan(1, 64, 2, 64, 2, 2, device="cpu", **rm).steps() == ["seq_to_head", "attn_partial", "merge",
                                                                        "head_to_seq"]
    with pytest.raises(ValueError):
        UspPlan(1, 64, 2, 64, 2, 2, device="cpu", ring_merge="tree")
    # the default: fold on 16-bit inputs at any ring degree, partials and
    # the merge on the fp32 path
    assert UspPlan(1, 64, 2, 64, 2, 4, device="cpu").ring_merge == "fold"
    assert UspPlan(1, 64, 2, 64, 2, 2, device="cpu", in_dtype=torch.float32).ring_merge == "partials"


def test_ring_rows_argument_checks(dl):
    """dit_attn_ring_rows refuses, before any launch: a NULL row array, a
    negative output row, and blocks whose output rows overlap in one tensor
    (o.stride_q == 0).  (Disjoint rows are run on the GPU, in test_gpu_ring.)"""
    from sequence_attention_gb300._lib import DitLseView, DitView
    L = dl.lib()
    H, D = 2, 128
    q = DitView()
    q.ptr, q.stride_q, q.stride_b, q.stride_s, q.stride_h = 1 << 20, 64 * H * D, 64 * H * D, H * D, D
    o = DitView()                        # one [1, 256, H, D] tensor for both blocks
    o.ptr, o.stride_b, o.stride_s, o.stride_h = 1 << 20, 256 * H * D, H * D, D
    lse = DitLseView()
    lens = (ctypes.c_int * 2)(64, 64)

    def call(rows):
        r = None if rows is None else (ctypes.c_int * 2)(*rows)
        return L.dit_attn_ring_rows(1, H, D, 0.1, 2, lens, r, 2, lens, q, dl.DIT_BF16, q, q, dl.DIT_F16, o,
                                    dl.DIT_BF16, lse, None, None)

    assert call(None) == dl.DIT_ERR_INVALID_ARG
    assert call([0, -1]) == dl.DIT_ERR_INVALID_ARG
    assert call([0, 32]) == dl.DIT_ERR_INVALID_ARG       # rows 32..63 written by both blocks
