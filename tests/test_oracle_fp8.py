"""Pins for the oracle's FP8 (e4m3) wire: the format against PyTorch's
float8_e4m3fn, ties and saturation from the format's definition, the error
bound of per-head scaling, and the exchange by brute-force indexing."""
import numpy as np
import torch

import synth
from oracle import fp8
from oracle import layout as olayout
from oracle import numeric
from tests.helpers import bits


def test_every_code_decodes_like_torch():
    c = np.arange(256, dtype=np.uint8)
    ours = fp8.e4m3_value(c)
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_encoding_matches_torch_in_range():
    rng = np.random.default_rng(0)
    y = np.concatenate([rng.standard_normal(50000) * 60, rng.standard_normal(20000) * 1e-3,
                        -rng.random(1000) * 2.0 ** -10, [0.0, -0.0]]).astype(np.float32)
    y = y[np.abs(y) < 464]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(fp8.e4m3_encode(y), ref)


def test_midpoints_round_to_the_even_code():
    codes = np.arange(0x7E, dtype=np.uint8)           # pairs (c, c+1) of finite codes
    v = fp8.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    mid = (v[:-1] + v[1:]) / 2                          # exact in float64
    want = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    np.testing.assert_array_equal(fp8.e4m3_encode(mid), want)
    np.testing.assert_array_equal(fp8.e4m3_encode(-mid), want | 0x80)


def test_saturation_and_nan():
    got = fp8.e4m3_encode(np.array([448.0, 460.0, 1000.0, 1e30, -1e30, np.inf, -np.inf, np.nan]))
    np.testing.assert_array_equal(got, [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE, 0x7F])


def test_head_scaling_bound_and_extremes():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 7, 128)) * np.exp2(rng.integers(-20, 20, (64, 7, 1)))).astype(np.float32)
    x[3, 2] = 0.0                                        # an all-zero head
    codes, s = fp8.quantize_heads(x)
    y = fp8.dequantize_heads(codes, s).astype(np.float64)
    # half an e4m3 ulp: 2^-4 relative in the normal range, 2^-10 * s below it
    bound = (2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s[..., None]) * (1 + 2.0 ** -20)
    assert np.all(np.abs(y - x) <= bound)
    # the largest magnitude of each non-zero head lands on +-448
    k = np.argmax(np.abs(x), axis=-1)
    top = np.take_along_axis(codes, k[..., None], -1)[..., 0]
    nz = s > 0
    assert np.all((top[nz] & 0x7F) == 0x7E)
    assert s[3, 2] == 0 and np.all(codes[3, 2] == 0) and np.all(y[3, 2] == 0)


def test_records_hold_codes_then_the_scale():
    codes = np.arange(32, dtype=np.uint8).reshape(2, 16)
    s = np.array([1.5, -0.25], dtype=np.float32)
    rec = fp8.to_records(codes, s)
    assert rec.shape == (2, 32) and np.all(rec[:, 20:] == 0)
    assert rec[0, 16:20].view(np.float32)[0] == 1.5
    c2, s2 = fp8.from_records(rec)
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(s2, s)


def test_exchange_delivers_each_heads_quantized_values():
    # brute force: rank (r, v)'s head layout = the quantized-dequantized
    # global planes, read straight from their rows and heads
    B, S, H, D, U, R = 2, 19, 5, 16, 3, 2
    L = olayout.make_layout(B, S, H, D, U, R)
    planes = [bits(synth.normal((B, S, H, D), 60 + p, 1.0, "bf16")) for p in range(2)]
    recv = fp8.a2a(L, "s2h", 2, fp8.s2h_pack(L, planes, "bf16"))
    got = fp8.s2h_unpack(L, recv, ["f32", "f32"])
    for p in range(2):
        x = numeric.to_f64(planes[p], "bf16").astype(np.float32)
        want = fp8.dequantize_heads(*fp8.quantize_heads(x))
        for (r, v), pl in got.items():
            for s_ in range(L.ring_len[r]):
                t = L.ring_off[r] + s_
                for hl in range(L.Hl):
                    h = v * L.Hl + hl
                    w = want[:, t, h] if h < H else np.zeros((B, D), np.float32)
                    np.testing.assert_array_equal(numeric.to_f64(pl[p][:, s_, hl], "f32"), w)


def test_head_to_seq_exchange_drops_padding():
    B, S, H, D, U, R = 1, 13, 5, 16, 3, 1
    L = olayout.make_layout(B, S, H, D, U, R)
    o = synth.normal((B, S, L.Hp, D), 70, 1.0, "f32").numpy()
    o_ranks = {(0, v): bits(torch.from_numpy(np.ascontiguousarray(o[:, :, v * L.Hl:(v + 1) * L.Hl])))
               for v in range(U)}
    recv = fp8.a2a(L, "h2s", 1, fp8.h2s_pack(L, o_ranks, "f32"))
    got = numeric.to_f64(fp8.h2s_unpack(L, recv, "f32"), "f32")
    want = fp8.dequantize_heads(*fp8.quantize_heads(o[:, :, :H]))
    np.testing.assert_array_equal(got, want)


def test_exchange_in_the_unpadded_and_lcm_padded_layouts():
    B, S, H, D, U, R = 1, 70, 5, 16, 3, 2
    for ph, pl in [(False, False), (True, True), (False, True)]:
        L = olayout.make_layout(B, S, H, D, U, R, pad_heads=ph, pad_lcm64=pl)
        x = bits(synth.normal((B, S, H, D), 80, 1.0, "bf16"))
        recv = fp8.a2a(L, "s2h", 1, fp8.s2h_pack(L, [x], "bf16"))
        want = fp8.dequantize_heads(*fp8.quantize_heads(numeric.to_f64(x, "bf16").astype(np.float32)))
        for (r, v), planes in fp8.s2h_unpack(L, recv, ["f32"]).items():
            got = numeric.to_f64(planes[0], "f32")
            m = L.real_rows(r)
            h0, h1 = L.head_off[v], min(L.head_off[v] + L.head_len[v], H)
            np.testing.assert_array_equal(got[:, :m, :h1 - h0], want[:, L.ring_off[r]:L.ring_off[r] + m, h0:h1])
            assert np.all(got[:, m:] == 0) and np.all(got[:, :, h1 - h0:] == 0)


def test_float32_step_order_agrees_with_the_exact_scale():
    """The pages fix no e4m3 format; the oracle reads it as float32 steps
    (amax, s = amax / 448, r = 1 / s, y = x * r, then the code).  Against the
    exact scale (y = x * 448 / amax in float64, then the same rounding) the
    codes agree, except where the exact y lies within a few float32 ulps of a
    midpoint between two codes; there they differ by one step."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((1024, 8, 128)) * np.exp2(rng.integers(-12, 12, (1024, 8, 1)))).astype(np.float32)
    codes, _ = fp8.quantize_heads(x)
    amax = np.abs(x.astype(np.float64)).max(axis=-1, keepdims=True)
    y = x.astype(np.float64) * (448.0 / amax)
    exact = fp8.e4m3_encode(y)
    diff = codes != exact
    assert diff.mean() <= 1e-4
    if diff.any():
        a, b = codes[diff], exact[diff]
        assert np.all((a >> 7) == (b >> 7))                      # same sign
        assert np.all(np.abs((a & 0x7F).astype(int) - (b & 0x7F).astype(int)) == 1)
        lo = np.minimum(fp8.e4m3_value(a & 0x7F), fp8.e4m3_value(b & 0x7F))
        hi = np.maximum(fp8.e4m3_value(a & 0x7F), fp8.e4m3_value(b & 0x7F))
        mid = (lo + hi) / 2
        assert np.all(np.abs(np.abs(y[diff]) - mid) <= 4 * 2.0 ** -23 * mid)
    # each non-zero head's largest magnitude is exactly 448 on both sides
    k = np.argmax(np.abs(x), axis=-1)[..., None]
    assert np.all((np.take_along_axis(codes, k, -1) & 0x7F) == 0x7E)
    assert np.all((np.take_along_axis(exact, k, -1) & 0x7F) == 0x7E)
