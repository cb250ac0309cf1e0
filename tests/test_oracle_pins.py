"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a value the pages print, a closed form, a
library routine (torch bf16 conversion, numpy complex arithmetic,
scipy.linalg.hadamard, torch scaled_dot_product_attention), an invariant of the
mathematics, or brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import torch
import torch.nn.functional as F

from oracle import v4_oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")))
RNG = np.random.default_rng(1234)


def unit_rms(x):
    return x / np.sqrt((x * x).mean(-1, keepdims=True))


def sdpa64(q, k, v, mask=None, scale=None):
    """torch SDPA in float64 on CPU. q [H,1,D] k/v [1?,nk,D]; mask additive or bool."""
    return F.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=None if mask is None else torch.from_numpy(mask), scale=scale).numpy()


# ----------------------------------------------------------------- rounding
def test_bf16_rounding_matches_torch():
    x = (RNG.standard_normal(20000) * np.exp(RNG.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x.astype(np.float64)), ref)


def test_bf16_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: even mantissa is 1.
    assert O.round_to_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6.
    assert O.round_to_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert O.round_to_bf16(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert O.round_to_bf16(0.0) == 0.0


# ----------------------------------------------------------------- RoPE
def test_inv_freq_closed_form_values():
    f = O.make_inv_freq(40000.0, 64)
    assert f.dtype == np.float32 and f.shape == (32,)
    assert f[0] == 1.0
    # pair j = R/4 has exponent -1/2: 40000^-1/2 = 1/200
    assert abs(float(f[16]) - 1.0 / 200.0) < 1e-9
    assert np.all(np.diff(f) < 0)


def test_yarn_boundary_behaviour():
    base = O.make_inv_freq(40000.0, 64).astype(np.float64)
    y = O.make_inv_freq(40000.0, 64, yarn_factor=16.0, original_len=4096).astype(np.float64)
    wl = 2 * math.pi / base
    r = 4096 / wl
    hi = r > 32.0       # high-frequency pairs are untouched
    lo = r < 1.0        # lowest-frequency pairs are fully interpolated (divided by s)
    assert hi.any() and lo.any()
    np.testing.assert_allclose(y[hi], base[hi], rtol=1e-7)
    np.testing.assert_allclose(y[lo], base[lo] / 16.0, rtol=1e-6)
    mid = ~(hi | lo)
    assert np.all((y[mid] <= base[mid] + 1e-12) & (y[mid] >= base[mid] / 16.0 - 1e-12))
    # factor 1 or no original length: identity
    np.testing.assert_array_equal(O.make_inv_freq(40000.0, 64, 1.0, 4096), O.make_inv_freq(40000.0, 64))
    np.testing.assert_array_equal(O.make_inv_freq(40000.0, 64, 16.0, 0), O.make_inv_freq(40000.0, 64))


def test_yarn_mscale_is_the_printed_factor():
    g = GOLD["yarn_mscale_not_applied"]
    assert abs(O.yarn_attention_mscale(16.0) - g["value"]) < 5e-4


def test_rope_is_complex_multiplication():
    D, R = 64, 16
    f = O.make_inv_freq(40000.0, R)
    x = RNG.standard_normal((5, D))
    pos = np.array([0, 3, 17, 255, 4096])
    y = O.rope_rotate(x, pos, f)
    np.testing.assert_array_equal(y[:, :D - R], x[:, :D - R])
    z = x[:, D - R::2] + 1j * x[:, D - R + 1::2]
    zr = z * np.exp(1j * pos[:, None] * f.astype(np.float64)[None, :])
    np.testing.assert_allclose(y[:, D - R::2], zr.real, atol=1e-13)
    np.testing.assert_allclose(y[:, D - R + 1::2], zr.imag, atol=1e-13)


def test_rope_roundtrip_and_norm():
    f = O.make_inv_freq(40000.0, 64, 16.0, 4096)
    x = RNG.standard_normal((7, 512))
    pos = RNG.integers(0, 1 << 20, 7)
    y = O.rope_rotate(x, pos, f)
    np.testing.assert_allclose(O.rope_derotate(y, pos, f), x, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-14)


@pytest.mark.parametrize("ratio", [4, 16, 128])
def test_rope_relative_position_with_compressed_positions(ratio):
    # The query at t and entry s at position ratio*s: the dot product depends on
    # t - ratio*s only.  Ratio > 1 is the case that separates "entry rotated at
    # s" from "entry rotated at ratio*s".
    f = O.make_inv_freq(40000.0, 64)
    q = RNG.standard_normal(512)
    k = RNG.standard_normal(512)
    s = 37
    t = ratio * s + 5
    a = O.rope_rotate(q, t, f) @ O.rope_rotate(k, ratio * s, f)
    b = O.rope_rotate(q, t - ratio * s, f) @ k
    assert abs(a - b) < 1e-10
    wrong = O.rope_rotate(q, t, f) @ O.rope_rotate(k, s, f)
    assert abs(wrong - a) > 1e-3


# ----------------------------------------------------------------- Hadamard
@pytest.mark.parametrize("n", [1, 2, 32, 128])
def test_hadamard_is_scipy_sylvester_and_orthogonal(n):
    h = O.hadamard_matrix(n)
    np.testing.assert_array_equal(h * math.sqrt(n), scipy.linalg.hadamard(n).astype(np.float64))
    np.testing.assert_allclose(h @ h.T, np.eye(n), atol=1e-14)


# ----------------------------------------------------------------- counting
def test_entry_counts_and_visibility():
    assert O.num_entries(16384, 4) == 4096 and O.num_entries(16384, 128) == 128
    assert O.num_entries(1003, 4) == 250          # partial trailing group is dropped
    assert [O.n_visible(t, 4) for t in range(9)] == [0, 0, 0, 1, 1, 1, 1, 2, 2]
    # brute force: entry s visible to t iff its last own token <= t
    for r in (1, 4, 128):
        for t in range(0, 600, 7):
            bf = sum(1 for s in range(1000) if r * s + r - 1 <= t)
            assert O.n_visible(t, r) == bf


def test_reads_per_query_at_one_million():
    g = GOLD["reads_per_query_at_1M"]
    t = g["context"] - 1
    assert O.keys_read(t, 4, 128, 512) == g["csa"]
    hca = O.keys_read(t, 128, 128, 0)
    assert hca == 1000000 // 128 + 128
    assert abs(hca - g["hca_roughly"]) / g["hca_roughly"] < 0.01


def test_pooling_window_sizes():
    g = GOLD["pooling_windows"]
    assert len(O.group_members(5, 4, 1)) == g["csa"]
    assert len(O.group_members(5, 128, 0)) == g["hca"]
    assert len(O.group_members(0, 4, 1)) == 4       # entry 0 has no previous group


# ----------------------------------------------------------------- compressor
def _comp_inputs(B, S, r, ov, d, score_std=1.0):
    ckv = unit_rms(RNG.standard_normal((B, S, 1 + ov, d)))
    cs = RNG.standard_normal((B, S, 1 + ov, d)) * score_std
    ape = RNG.standard_normal(((1 + ov) * r, d)) * 0.1
    return ckv, cs, ape


def test_pooling_weights_sum_to_one():
    ckv, cs, ape = _comp_inputs(2, 40, 4, 1, 16)
    for s in (0, 1, 9):
        _, w = O.pooling_weights(cs, ape, s, 4, 1)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-14)
        assert np.all(w > 0)


def test_constant_score_gives_mean_of_members():
    B, S, r, d = 1, 32, 4, 16
    ckv = RNG.standard_normal((B, S, 2, d))
    cs = np.full((B, S, 2, d), 0.3)
    ape = np.zeros((2 * r, d))
    f = O.make_inv_freq(40000.0, 4)
    e = O.compress(ckv, cs, ape, None, f, r, 1, 0.0)
    for s in (0, 3, 7):
        mem = O.group_members(s, r, 1)
        mean = np.mean([ckv[0, j, h] for (j, h, _) in mem], axis=0)
        ref = mean / np.sqrt((mean ** 2).mean())
        ref = O.rope_rotate(ref, r * s, f)
        np.testing.assert_allclose(e[0, s], ref, atol=1e-12)


def test_ratio_one_no_overlap_is_normed_rotated_token():
    B, S, d = 2, 12, 32
    ckv, cs, ape = _comp_inputs(B, S, 1, 0, d)
    g = RNG.uniform(0.5, 1.5, d)
    f = O.make_inv_freq(10000.0, 8)
    e = O.compress(ckv, cs, ape, g, f, 1, 0, 1e-6)
    x = ckv[:, :, 0, :]
    ref = x / np.sqrt((x * x).mean(-1, keepdims=True) + 1e-6) * g
    ref = O.rope_rotate(ref, np.arange(S)[None, :], f)
    np.testing.assert_allclose(e, ref, atol=1e-12)


def test_one_hot_score_selects_member():
    B, S, r, d = 1, 24, 4, 8
    ckv, cs, ape = _comp_inputs(B, S, r, 1, d)
    cs[:] = 0.0
    ape[:] = 0.0
    # entry 3: make the previous group's member i=2 (token 10, half 1) dominate
    cs[0, 10, 1, :] = 1000.0
    f = O.make_inv_freq(40000.0, 4)
    e = O.compress(ckv, cs, ape, None, f, r, 1, 0.0)
    x = ckv[0, 10, 1]
    ref = O.rope_rotate(x / np.sqrt((x * x).mean()), 12, f)
    np.testing.assert_allclose(e[0, 3], ref, atol=1e-12)


def test_ape_row_order_is_chronological():
    # with zero scores, ape alone chooses the member: a huge bias on row 0 picks
    # the oldest token of the previous group, on row r the first own token.
    B, S, r, d = 1, 16, 4, 8
    ckv, cs, ape = _comp_inputs(B, S, r, 1, d)
    cs[:] = 0.0
    f = O.make_inv_freq(40000.0, 4)
    for row, token, half in ((0, 4, 1), (r, 8, 0), (2 * r - 1, 11, 0)):
        ape[:] = 0.0
        ape[row, :] = 1000.0
        e = O.compress(ckv, cs, ape, None, f, r, 1, 0.0)
        x = ckv[0, token, half]
        ref = O.rope_rotate(x / np.sqrt((x * x).mean()), 2 * r, f)
        np.testing.assert_allclose(e[0, 2], ref, atol=1e-12)


def test_scalar_score_equals_broadcast_channel_score():
    B, S, r, d = 1, 20, 4, 8
    ckv, _, ape = _comp_inputs(B, S, r, 1, d)
    ape[:] = 0.0
    scal = RNG.standard_normal((B, S, 2, 1))
    f = O.make_inv_freq(40000.0, 4)
    e = O.compress(ckv, np.broadcast_to(scal, (B, S, 2, d)), ape, None, f, r, 1, 1e-6)
    # reference: token-level softmax weights applied to whole rows
    for s in range(S // r):
        mem = O.group_members(s, r, 1)
        lam = np.array([scal[0, j, h, 0] for (j, h, _) in mem])
        wts = np.exp(lam - lam.max())
        wts /= wts.sum()
        pooled = sum(wt * ckv[0, j, h] for wt, (j, h, _) in zip(wts, mem))
        ref = O.rope_rotate(pooled / np.sqrt((pooled ** 2).mean() + 1e-6), r * s, f)
        np.testing.assert_allclose(e[0, s], ref, atol=1e-12)


def test_entry_zero_excludes_missing_previous_group():
    B, S, r, d = 1, 8, 4, 8
    ckv, cs, ape = _comp_inputs(B, S, r, 1, d)
    f = O.make_inv_freq(40000.0, 4)
    e = O.compress(ckv, cs, ape, None, f, r, 1, 0.0)
    lam = cs[0, 0:4, 0] + ape[4:8]
    wts = np.exp(lam - lam.max(0))
    wts /= wts.sum(0)
    pooled = (wts * ckv[0, 0:4, 0]).sum(0)
    ref = O.rope_rotate(pooled / np.sqrt((pooled ** 2).mean()), 0, f)
    np.testing.assert_allclose(e[0, 0], ref, atol=1e-12)


# ----------------------------------------------------------------- indexer
def test_indexer_temperature_is_printed_constant():
    g = GOLD["indexer_temperature_inverse"]
    c = O.indexer_scale(g["at"]["idx_heads"], g["at"]["idx_dim"])
    assert abs(1.0 / c - g["value"]) < 0.05
    assert c == 1.0 / math.sqrt(64 * 128)


def test_indexer_scores_invariant_under_hadamard():
    # prep (rotation + Hadamard on both sides) gives the same scores as the
    # plain rotated dot products: the Hadamard is orthogonal.
    B, S, Hi, Di, r = 1, 64, 3, 32, 4
    f = O.make_inv_freq(40000.0, 16)
    iq = RNG.standard_normal((B, S, Hi, Di))
    ickv, ics, iape = _comp_inputs(B, S, r, 1, Di)
    w = RNG.standard_normal((B, S, Hi))
    ikey = O.compress(ickv, ics, iape, None, f, r, 1, 1e-6, hadamard=True)
    sc = O.indexer_scores(O.indexer_query_prep(iq, f), ikey, w, r)
    key_nh = O.compress(ickv, ics, iape, None, f, r, 1, 1e-6, hadamard=False)
    c = 1.0 / math.sqrt(Hi * Di)
    for t in (3, 17, 63):
        nv = O.n_visible(t, r)
        qr = O.rope_rotate(iq[0, t], t, f)
        ref = [sum(w[0, t, h] * c * max(0.0, qr[h] @ key_nh[0, s]) for h in range(Hi)) for s in range(nv)]
        np.testing.assert_allclose(sc[0, t, :nv], ref, rtol=1e-12, atol=1e-12)
        assert np.all(np.isneginf(sc[0, t, nv:]))


def test_topk_matches_brute_force_sort():
    for trial in range(20):
        n = int(RNG.integers(1, 60))
        k = int(RNG.integers(1, 20))
        row = np.round(RNG.standard_normal(n), 1)   # rounding makes ties common
        idx, val = O.topk_select(row, n, k)
        ref = sorted(range(n), key=lambda s: (-row[s], s))[:k]
        assert list(idx[:len(ref)]) == ref
        assert np.all(idx[len(ref):] == -1)
        # every kept entry beats or ties every dropped one
        kept = set(ref)
        if len(ref) < n:
            assert min(row[list(kept)]) >= max(row[[s for s in range(n) if s not in kept]])


def test_topk_keeps_everything_when_k_covers_visible():
    B, S, Hi, Di, r, K = 1, 40, 2, 16, 4, 64
    f = O.make_inv_freq(40000.0, 4)
    iq = RNG.standard_normal((B, S, Hi, Di))
    ikey = RNG.standard_normal((B, S // r, Di))
    w = RNG.standard_normal((B, S, Hi))
    res = O.indexer_topk(iq, ikey, w, f, r, K)
    for t in range(S):
        nv = O.n_visible(t, r)
        got = res["idx"][0, t]
        assert sorted(got[got >= 0]) == list(range(nv))


# ----------------------------------------------------------------- attention
def _mqa_inputs(B, S, H, D):
    q = unit_rms(RNG.standard_normal((B, S, H, D)))
    kv = unit_rms(RNG.standard_normal((B, S, D)))
    return q, kv


def test_softmax_scale_is_head_dim_power():
    # One query, two keys with hand-set logits: o = softmax-weighted keys with
    # scale D^-1/2.  The YaRN-inflated scale (x1.277) gives a different answer.
    D, R = 512, 64
    f = np.zeros(R // 2, dtype=np.float32)         # no rotation
    q = np.zeros((1, 2, 1, D))
    kv = np.zeros((1, 2, D))
    q[0, 1, 0, 0] = 3.0
    kv[0, 0, 0] = 4.0
    kv[0, 1, 1] = 5.0        # q . k1 = 12, q . k2 = 0
    o, lse = O.sparse_mqa(q, kv, None, None, None, f, 0, 2, rows=[1])
    l1, l2 = 12.0 / math.sqrt(D), 0.0
    p1 = math.exp(l1) / (math.exp(l1) + math.exp(l2))
    assert abs(o[0, 0, 0, 0] - 4.0 * p1) < 1e-14
    assert abs(o[0, 0, 0, 1] - 5.0 * (1 - p1)) < 1e-14
    assert abs(lse[0, 0, 0] - math.log(math.exp(l1) + 1.0)) < 1e-14
    l1w = l1 * O.yarn_attention_mscale(16.0)
    p1w = math.exp(l1w) / (math.exp(l1w) + 1.0)
    assert abs(4.0 * p1w - o[0, 0, 0, 0]) > 1e-3


def _sdpa_reference(q, keys, mask, t, f, scale):
    """SDPA over (already rotated) keys for query t, then de-rotation."""
    H, D = q.shape
    qr = O.rope_rotate(q, t, f)[:, None, :]                 # [H,1,D]
    out = sdpa64(qr, keys[None], keys[None], mask[None, None, :], scale)[:, 0, :]
    return O.rope_derotate(out, t, f)


def test_hca_equals_dense_masked_sdpa():
    B, S, H, D, R, r, W = 1, 300, 3, 32, 8, 16, 20
    f = O.make_inv_freq(40000.0, R)
    q, kv = _mqa_inputs(B, S, H, D)
    ent = unit_rms(RNG.standard_normal((B, S // r, D)))
    rows = [0, 15, 16, 100, 299]
    o, _ = O.sparse_mqa(q, kv, ent, None, None, f, r, W, rows=rows)
    allkeys = np.concatenate([ent[0], O.rope_rotate(kv[0], np.arange(S), f)], 0)
    N = ent.shape[1]
    for i, t in enumerate(rows):
        mask = np.zeros(N + S, dtype=bool)
        mask[:O.n_visible(t, r)] = True
        mask[N + max(0, t - W + 1):N + t + 1] = True
        ref = _sdpa_reference(q[0, t], allkeys, mask, t, f, D ** -0.5)
        np.testing.assert_allclose(o[0, i], ref, atol=1e-12)


def test_csa_selection_equals_masked_sdpa():
    B, S, H, D, R, r, W, K = 1, 200, 4, 32, 8, 4, 16, 10
    f = O.make_inv_freq(40000.0, R)
    q, kv = _mqa_inputs(B, S, H, D)
    N = S // r
    ent = unit_rms(RNG.standard_normal((B, N, D)))
    idx = np.full((B, S, K), -1, dtype=np.int32)
    for t in range(S):
        nv = O.n_visible(t, r)
        take = min(K, nv)
        idx[0, t, RNG.permutation(K)[:take]] = RNG.permutation(nv)[:take]
    rows = [2, 3, 40, 199]
    o, lse = O.sparse_mqa(q, kv, ent, idx, None, f, r, W, rows=rows)
    allkeys = np.concatenate([ent[0], O.rope_rotate(kv[0], np.arange(S), f)], 0)
    for i, t in enumerate(rows):
        mask = np.zeros(N + S, dtype=bool)
        sel = idx[0, t][idx[0, t] >= 0]
        mask[sel] = True
        mask[N + max(0, t - W + 1):N + t + 1] = True
        ref = _sdpa_reference(q[0, t], allkeys, mask, t, f, D ** -0.5)
        np.testing.assert_allclose(o[0, i], ref, atol=1e-12)
        # lse against torch.logsumexp of the masked logits
        qr = O.rope_rotate(q[0, t], t, f)
        lg = torch.from_numpy((qr @ allkeys[mask].T) * D ** -0.5)
        np.testing.assert_allclose(lse[0, i], torch.logsumexp(lg, -1).numpy(), atol=1e-12)


@pytest.mark.parametrize("window", [-1, 0])
def test_ratio_one_layer_reduces_to_causal_mqa(window):
    # ratio 1, no overlap, no selection, ape 0, eps 0, pre-normalised tokens:
    # entry s equals the rotated token s.  With an unlimited window every token
    # is a key twice with the same value; duplicates cancel in the softmax and
    # the result is plain causal MQA over K = V = rot(kv).  With window 0 each
    # token is a key once, through its entry.
    B, S, H, D, R = 1, 48, 4, 32, 8
    f = O.make_inv_freq(10000.0, R)
    q, kv = _mqa_inputs(B, S, H, D)
    x = dict(q=q, kv=kv, ckv=kv[:, :, None, :], cscore=RNG.standard_normal((B, S, 1, D)),
             ape=np.zeros((1, D)), norm_w=None, inv_freq=f, sink=None)
    res = O.attn_layer(dict(ratio=1, overlap=0, window=window, topk=0, rms_eps=0.0), x)
    keys = O.rope_rotate(kv[0], np.arange(S), f)
    qr = np.stack([O.rope_rotate(q[0, t], t, f) for t in range(S)])       # [S,H,D]
    ref = F.scaled_dot_product_attention(
        torch.from_numpy(qr.transpose(1, 0, 2)), torch.from_numpy(keys)[None].expand(H, S, D),
        torch.from_numpy(keys)[None].expand(H, S, D), is_causal=True).numpy().transpose(1, 0, 2)
    ref = np.stack([O.rope_derotate(ref[t], t, f) for t in range(S)])
    np.testing.assert_allclose(res["o"][0], ref, atol=1e-12)


def test_sink_is_an_extra_zero_valued_key():
    B, S, H, D, R, W = 1, 30, 4, 32, 8, 8
    f = O.make_inv_freq(10000.0, R)
    q, kv = _mqa_inputs(B, S, H, D)
    z = RNG.standard_normal(H)
    rows = [0, 5, 29]
    o, lse = O.sparse_mqa(q, kv, None, None, z, f, 0, W, rows=rows)
    for i, t in enumerate(rows):
        lo = max(0, t - W + 1)
        keys = O.rope_rotate(kv[0, lo:t + 1], np.arange(lo, t + 1), f)
        keys0 = np.concatenate([keys, np.zeros((1, D))], 0)               # extra zero key
        qr = O.rope_rotate(q[0, t], t, f)[:, None, :]
        mask = np.zeros((H, 1, keys0.shape[0]))
        mask[:, 0, -1] = z                                                # its logit is z_h
        out = F.scaled_dot_product_attention(
            torch.from_numpy(qr), torch.from_numpy(keys0)[None].expand(H, -1, -1),
            torch.from_numpy(keys0)[None].expand(H, -1, -1),
            attn_mask=torch.from_numpy(mask), scale=D ** -0.5).numpy()[:, 0, :]
        np.testing.assert_allclose(o[0, i], O.rope_derotate(out, t, f), atol=1e-12)
    # a sink of -inf is no sink
    o2, _ = O.sparse_mqa(q, kv, None, None, np.full(H, -np.inf), f, 0, W, rows=rows)
    o3, _ = O.sparse_mqa(q, kv, None, None, None, f, 0, W, rows=rows)
    np.testing.assert_allclose(o2, o3, atol=0)


def test_single_key_derotation_returns_the_token():
    # window 1, no entries: o = derot(rot(kv[t], t), t) = kv[t]
    B, S, H, D, R = 1, 50, 3, 64, 16
    f = O.make_inv_freq(40000.0, R, 16.0, 4096)
    q, kv = _mqa_inputs(B, S, H, D)
    o, _ = O.sparse_mqa(q, kv, None, None, None, f, 0, 1)
    np.testing.assert_allclose(o[0], np.broadcast_to(kv[0][:, None, :], (S, H, D)), atol=1e-13)


def test_empty_key_set():
    B, S, H, D = 1, 6, 2, 16
    f = O.make_inv_freq(10000.0, 4)
    q, kv = _mqa_inputs(B, S, H, D)
    o, lse = O.sparse_mqa(q, kv, None, None, None, f, 4, 0)   # no window, no entries yet
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    z = np.array([0.5, -1.0])
    o, lse = O.sparse_mqa(q, kv, None, None, z, f, 4, 0)
    assert np.all(o == 0)
    np.testing.assert_allclose(lse[0], np.broadcast_to(z, (S, H)))


def test_grouped_wo_a_matches_per_group_matmul():
    B, T, H, D, G, rank = 2, 3, 8, 16, 4, 5
    o = RNG.standard_normal((B, T, H, D))
    wa = RNG.standard_normal((G, (H // G) * D, rank))
    y = O.grouped_wo_a(o, wa)
    for g in range(G):
        xg = torch.from_numpy(o[:, :, 2 * g:2 * g + 2, :].reshape(B, T, -1))
        ref = torch.matmul(xg, torch.from_numpy(wa[g])).numpy()
        np.testing.assert_allclose(y[:, :, g * rank:(g + 1) * rank], ref, atol=1e-12)


def test_flash_layer_mix():
    import seeded_inputs as SI
    g = GOLD["flash_layer_mix"]
    ratios = SI.flash_layer_ratios()
    assert len(ratios) == g["decoder_layers"]
    assert ratios.count(0) == g["swa"] and ratios.count(4) == g["csa"] and ratios.count(128) == g["hca"]
    assert ratios[-1] == 4 and ratios[:2] == [0, 0]


# ---------------------------------------------------------------------------
# Query projections from the shared rank-r latent
# ---------------------------------------------------------------------------
def _qproj_case(seed=0, B=2, T=5, r=16, H=3, D=8):
    rng = np.random.default_rng(seed)
    return rng.normal(0, 1, (B, T, r)), rng.normal(0, 0.3, (r, H * D)), H, D


def test_q_projection_matches_explicit_sums():
    qlat, wq, H, D = _qproj_case()
    y = O.q_projection(qlat, wq, H, D, norm=False)
    for (b, t, h, d) in ((0, 0, 0, 0), (1, 4, 2, 7), (0, 3, 1, 5)):
        ref = sum(qlat[b, t, k] * wq[k, h * D + d] for k in range(qlat.shape[-1]))
        assert abs(y[b, t, h, d] - ref) < 1e-12
    g = np.random.default_rng(1).normal(0, 1, D)
    yn = O.q_projection(qlat, wq, H, D, norm=True, eps=1e-6, norm_w=g)
    for (b, t, h) in ((0, 0, 0), (1, 4, 2)):
        v = y[b, t, h]
        ref = v / math.sqrt(sum(x * x for x in v) / D + 1e-6) * g
        np.testing.assert_allclose(yn[b, t, h], ref, rtol=1e-12, atol=1e-14)


def test_q_projection_heads_have_unit_rms_and_ignore_scale():
    qlat, wq, H, D = _qproj_case(2)
    y = O.q_projection(qlat, wq, H, D, norm=True)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-12)
    # each head is normalised on its own: scaling one head's weight columns
    # leaves every head unchanged
    w2 = wq.copy()
    w2[:, D:2 * D] *= 7.0
    np.testing.assert_allclose(O.q_projection(qlat, w2, H, D, norm=True), y, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(O.q_projection(3.0 * qlat, wq, H, D, norm=True), y, rtol=1e-12, atol=1e-14)


def test_indexer_q_projection_shares_the_latent():
    qlat, _, _, _ = _qproj_case(3)
    wiq = np.random.default_rng(4).normal(0, 0.3, (qlat.shape[-1], 2 * 4))
    y = O.indexer_q_projection(qlat, wiq, 2, 4)
    np.testing.assert_allclose(y.reshape(2, 5, 8), np.einsum("btk,kn->btn", qlat, wiq), rtol=1e-12)
    assert y.shape == (2, 5, 2, 4)
