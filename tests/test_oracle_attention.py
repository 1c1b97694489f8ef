"""Pins for the oracle's attention, partial and log-sum-exp merge.

Each check rests on something other than the oracle's own formula: closed
forms, invariances that any correct softmax attention has, and PyTorch's
scaled_dot_product_attention (a library routine) in float64.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as att


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, scale):
    """torch SDPA in float64, inputs [B,S,H,D] -> [B,Sq,H,D]."""
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


def test_zero_queries_give_mean_of_values():
    v = _rand((2, 9, 3, 5), 1)
    k = _rand((2, 9, 3, 5), 2)
    q = np.zeros((2, 4, 3, 5))
    o, lse = att.attention(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape),
                               rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(9.0), rtol=0, atol=1e-14)


def test_constant_values_pass_through():
    q, k = _rand((1, 6, 2, 4), 3), _rand((1, 11, 2, 4), 4)
    v = np.empty((1, 11, 2, 4))
    v[..., 0, :] = [0.5, -2.0, 3.0, 7.25]
    v[..., 1, :] = [1.0, 1.0, -1.0, 0.0]
    o, _ = att.attention(q, k, v)
    np.testing.assert_allclose(o[0, :, 0, :], np.broadcast_to(v[0, 0, 0], (6, 4)), atol=1e-14)
    np.testing.assert_allclose(o[0, :, 1, :], np.broadcast_to(v[0, 0, 1], (6, 4)), atol=1e-14)


def test_single_key():
    q, k, v = _rand((1, 5, 2, 8), 5), _rand((1, 1, 2, 8), 6), _rand((1, 1, 2, 8), 7)
    o, lse = att.attention(q, k, v, scale=0.3)
    for h in range(2):
        np.testing.assert_allclose(o[0, :, h], np.broadcast_to(v[0, 0, h], (5, 8)), atol=1e-15)
        np.testing.assert_allclose(lse[0, h], 0.3 * q[0, :, h] @ k[0, 0, h], atol=1e-14)


def test_two_keys_logistic_closed_form():
    q, k, v = _rand((1, 7, 1, 3), 8), _rand((1, 2, 1, 3), 9), _rand((1, 2, 1, 3), 10)
    sc = 0.7
    o, lse = att.attention(q, k, v, scale=sc)
    s0 = sc * q[0, :, 0] @ k[0, 0, 0]
    s1 = sc * q[0, :, 0] @ k[0, 1, 0]
    w0 = 1.0 / (1.0 + np.exp(s1 - s0))
    expect = w0[:, None] * v[0, 0, 0] + (1 - w0)[:, None] * v[0, 1, 0]
    np.testing.assert_allclose(o[0, :, 0], expect, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], np.logaddexp(s0, s1), atol=1e-14)


@pytest.mark.parametrize("B,Sq,Sk,H,D", [(1, 5, 13, 3, 8), (2, 17, 4, 2, 16), (1, 1, 1, 1, 1)])
def test_output_matches_torch_sdpa(B, Sq, Sk, H, D):
    q, k, v = _rand((B, Sq, H, D), 11), _rand((B, Sk, H, D), 12), _rand((B, Sk, H, D), 13)
    for scale in (None, 0.25):
        sc = 1.0 / math.sqrt(D) if scale is None else scale
        o, _ = att.attention(q, k, v, scale=scale)
        np.testing.assert_allclose(o, _sdpa(q, k, v, sc), rtol=1e-12, atol=1e-13)


def test_lse_through_a_zero_key_probe():
    # Append a zero key (score 0 for every query) and read its softmax weight
    # from torch SDPA with an indicator value column: p* = exp(-lse').  The
    # original lse is ln(exp(lse') - 1).
    B, Sq, Sk, H, D = 1, 6, 10, 2, 8
    q, k = _rand((B, Sq, H, D), 14), _rand((B, Sk, H, D), 15)
    k2 = np.concatenate([k, np.zeros((B, 1, H, D))], axis=1)
    ind = np.zeros((B, Sk + 1, H, D))
    ind[:, Sk, :, 0] = 1.0
    p_star = _sdpa(q, k2, ind, 1.0 / math.sqrt(D))[..., 0]       # [B,Sq,H]
    lse_aug = -np.log(p_star)
    lse_expect = np.log(np.expm1(lse_aug)).transpose(0, 2, 1)
    _, lse = att.attention(q, k, np.zeros((B, Sk, H, D)))
    np.testing.assert_allclose(lse, lse_expect, rtol=1e-11, atol=1e-11)


def test_key_shift_invariance():
    # Adding w to every key adds scale*q.w to a whole score row: O unchanged,
    # lse shifted by exactly that amount.  Catches a softmax over the wrong axis.
    q, k, v = _rand((1, 8, 2, 6), 16), _rand((1, 12, 2, 6), 17), _rand((1, 12, 2, 6), 18)
    w = _rand((6,), 19)
    o1, l1 = att.attention(q, k, v)
    o2, l2 = att.attention(q, k + w, v)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    shift = (q @ w / math.sqrt(6)).transpose(0, 2, 1)
    np.testing.assert_allclose(l2 - l1, shift, atol=1e-12)


def test_key_permutation_invariance_and_head_independence():
    q, k, v = _rand((1, 5, 3, 4), 20), _rand((1, 9, 3, 4), 21), _rand((1, 9, 3, 4), 22)
    perm = np.random.default_rng(23).permutation(9)
    o1, l1 = att.attention(q, k, v)
    o2, l2 = att.attention(q, k[:, perm], v[:, perm])
    np.testing.assert_allclose(o2, o1, atol=1e-14)
    np.testing.assert_allclose(l2, l1, atol=1e-14)
    # Changing head 1's keys (a rescale, not a shift) leaves heads 0 and 2
    # untouched.
    k3 = k.copy()
    k3[:, :, 1] *= 3.0
    o3, _ = att.attention(q, k3, v)
    np.testing.assert_array_equal(o3[:, :, [0, 2]], o1[:, :, [0, 2]])
    assert not np.allclose(o3[:, :, 1], o1[:, :, 1])


def test_partial_excludes_padding_rows():
    q = _rand((1, 4, 2, 8), 24)
    k, v = _rand((1, 16, 2, 8), 25), _rand((1, 16, 2, 8), 26)
    kp, vp = k.copy(), v.copy()
    kp[:, 11:] = np.nan
    vp[:, 11:] = np.nan
    o, lse = att.partial(q, kp, vp, 11)
    o_ref, lse_ref = att.attention(q, k[:, :11], v[:, :11])
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(lse, lse_ref)


def test_empty_chunk():
    q = _rand((1, 3, 2, 4), 27)
    o, lse = att.partial(q, _rand((1, 5, 2, 4), 28), _rand((1, 5, 2, 4), 29), 0)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("cuts", [[0, 37], [0, 10, 37], [0, 1, 2, 30, 37], [0, 0, 20, 20, 37]])
def test_merge_of_any_partition_equals_single_shot(cuts):
    q, k, v = _rand((2, 6, 3, 8), 30), _rand((2, 37, 3, 8), 31), _rand((2, 37, 3, 8), 32)
    parts = [att.partial(q, k[:, a:b], v[:, a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = att.merge(parts)
    o_ref, lse_ref = att.attention(q, k, v)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)
    # Order of the parts does not matter.
    o2, lse2 = att.merge(parts[::-1])
    np.testing.assert_allclose(o2, o, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, atol=1e-14)


def test_partial_lies_between_the_values_it_averages():
    """A chunk-normalised partial is a convex combination of the chunk's V
    rows: every element lies between that column's smallest and largest
    value (so it cannot leave V's range, whatever its storage type).  A
    missing or wrong normalisation fails this."""
    q = _rand((2, 9, 3, 8), 80) * 4.0
    k = _rand((2, 40, 3, 8), 81) * 4.0
    v = _rand((2, 40, 3, 8), 82) * 3.0e4
    for a, b in ((0, 40), (5, 6), (7, 33)):
        o, _ = att.partial(q, k[:, a:b], v[:, a:b])
        lo = v[:, a:b].min(axis=1, keepdims=True)
        hi = v[:, a:b].max(axis=1, keepdims=True)
        slack = 1e-12 * np.abs(v).max()
        assert np.all(o >= lo - slack) and np.all(o <= hi + slack)


def test_merge_of_one_part_is_identity():
    q, k, v = _rand((1, 4, 2, 8), 33), _rand((1, 9, 2, 8), 34), _rand((1, 9, 2, 8), 35)
    p = att.attention(q, k, v)
    o, lse = att.merge([p])
    np.testing.assert_array_equal(o, p[0])
    np.testing.assert_array_equal(lse, p[1])


def test_merge_all_empty():
    q = _rand((1, 3, 1, 4), 36)
    e = att.partial(q, np.zeros((1, 2, 1, 4)), np.zeros((1, 2, 1, 4)), 0)
    o, lse = att.merge([e, e])
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_merge_rescales_with_the_right_sign():
    # Two chunks whose lse differ by ln 3: the merged O is (3*O_a + O_b)/4
    # when lse_a = lse_b + ln 3.  A sign slip in exp(lse_r - lse) fails this.
    oa = np.full((1, 1, 1, 2), 1.0)
    ob = np.full((1, 1, 1, 2), 5.0)
    la = np.array([[[math.log(3.0) + 0.2]]])
    lb = np.array([[[0.2]]])
    o, lse = att.merge([(oa, la), (ob, lb)])
    np.testing.assert_allclose(o, 2.0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.2 + math.log(4.0), atol=1e-15)


def test_masked_with_every_key_allowed_is_attention():
    rng = np.random.default_rng(40)
    q, k, v = (rng.standard_normal((2, 9, 3, 8)) for _ in range(3))
    o, l = att.masked(q, k, v, np.ones((2, 9), bool))
    o2, l2 = att.attention(q, k, v)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(l, l2, atol=1e-14)


def test_masked_equals_attention_over_the_gathered_keys():
    # the tail-padded text path: keys [txt_len, S_txt) of each batch are padding
    rng = np.random.default_rng(41)
    B, S, H, D, S_txt = 2, 20, 2, 8, 7
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    txt_len = [4, 7]
    mask = np.ones((B, S), bool)
    for b in range(B):
        mask[b, txt_len[b]:S_txt] = False
    o, l = att.masked(q, k, v, mask)
    for b in range(B):
        keep = np.flatnonzero(mask[b])
        o2, l2 = att.attention(q[b:b + 1], k[b:b + 1, keep], v[b:b + 1, keep])
        np.testing.assert_allclose(o[b], o2[0], atol=1e-14)
        np.testing.assert_allclose(l[b], l2[0], atol=1e-14)


def test_masked_text_is_the_merge_of_its_two_key_ranges():
    # the pages fold the masked text portion into the rest with the same merge
    rng = np.random.default_rng(42)
    B, S, H, D, S_txt, txt_len = 1, 30, 2, 8, 10, 6
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    mask = np.ones((B, S), bool)
    mask[:, txt_len:S_txt] = False
    o, l = att.masked(q, k, v, mask)
    parts = [att.partial(q, k[:, :S_txt], v[:, :S_txt], txt_len), att.attention(q, k[:, S_txt:], v[:, S_txt:])]
    o2, l2 = att.merge(parts)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(l, l2, atol=1e-13)


def test_masked_row_without_keys_is_empty():
    q = np.ones((1, 2, 1, 4))
    mask = np.array([[[True, False], [False, False]]])
    o, l = att.masked(q, q, q, mask)
    assert np.all(o[0, 1] == 0) and np.isneginf(l[0, 0, 1]) and np.isfinite(l[0, 0, 0])


def test_varlen_is_block_diagonal_masked_attention():
    rng = np.random.default_rng(43)
    cu_q, cu_k = [0, 3, 3, 10, 16], [0, 5, 9, 9, 20]      # an empty query segment and an empty key one
    Tq, Tk, H, D = cu_q[-1], cu_k[-1], 2, 8
    q = rng.standard_normal((Tq, H, D))
    k, v = rng.standard_normal((Tk, H, D)), rng.standard_normal((Tk, H, D))
    o, l = att.varlen(q, k, v, cu_q, cu_k)
    mask = np.zeros((1, Tq, Tk), bool)
    for s in range(4):
        mask[0, cu_q[s]:cu_q[s + 1], cu_k[s]:cu_k[s + 1]] = True
    o2, l2 = att.masked(q[None], k[None], v[None], mask)
    np.testing.assert_allclose(o, o2[0], atol=1e-14)
    np.testing.assert_allclose(l, l2[0], atol=1e-14)
    assert np.all(o[3:10] == 0)                          # the sequence whose keys are empty
