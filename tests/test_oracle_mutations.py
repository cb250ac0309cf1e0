"""Plant plausible mistakes in the oracle (CPU only) and check a pin catches each.

Every mutation is applied with monkeypatch to the oracle module, one pin test is
run against the mutated oracle, and that pin must fail.
"""
import math

import numpy as np
import pytest

from oracle import v4_oracle as O
import tests.test_oracle_fp8_pins as F
import tests.test_oracle_kl_pins as KL
import tests.test_oracle_pins as P

_rope = O.rope_rotate
_mqa = O.sparse_mqa
_had = O.hadamard_matrix
_pw = O.pooling_weights
_win = O.window_range
_comp = O.compress


def _flip_sign(x, pos, f):
    return _rope(x, -np.asarray(pos, dtype=np.float64), f)


def _inflated_scale(q, kv, ent, idx, sink, f, r, W, scale=None, **kw):
    D = np.asarray(q).shape[-1]
    return _mqa(q, kv, ent, idx, sink, f, r, W, scale=D ** -0.5 * O.yarn_attention_mscale(16.0), **kw)


def _ties_high(row, nvis, k):
    idx = np.full(k, -1, dtype=np.int32)
    val = np.full(k, -np.inf)
    if nvis <= 0:
        return idx, val
    s = np.arange(nvis)
    order = np.lexsort((-s, -np.asarray(row[:nvis])))[:min(k, nvis)]
    idx[:len(order)] = order
    val[:len(order)] = row[order]
    return idx, val


def _no_ape(cscore, ape, s, r, ov):
    return _pw(cscore, np.zeros_like(ape), s, r, ov)


def _window_off_by_one(t, W):
    lo, hi = _win(t, W)
    return (lo, hi - 1) if hi > lo else (lo, hi)


def _unnormalised_hadamard(n):
    return _had(n) * math.sqrt(n)


def _rotate_at_entry_index(ckv, cscore, ape, g, f, r, ov, eps, hadamard=False, store_bf16=False):
    # rotate entries at s instead of r*s: undo r*s rotation then rotate at s
    e = _comp(ckv, cscore, ape, g, f, r, ov, eps, hadamard=False, store_bf16=False)
    N = e.shape[1]
    e = O.rope_rotate(O.rope_derotate(e, (r * np.arange(N))[None, :], f), np.arange(N)[None, :], f)
    if hadamard:
        e = e @ _had(e.shape[-1]).T
    return O.maybe_bf16(e, store_bf16)


_e4m3 = O.round_to_e4m3
_quant = O.quantize_e4m3_rows


def _e4m3_two_mantissa_bits(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(ex - 1, -6) - 2)
    return np.copysign(np.minimum(np.rint(a / q) * q, 448.0), x)


def _e4m3_half_up(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    return np.copysign(np.minimum(np.floor(a / q + 0.5) * q, 448.0), x)


def _e4m3_no_saturation(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    return np.copysign(np.rint(a / q) * q, x)


def _quant_inverted_scale(x):
    codes, scales = _quant(x)
    return codes, np.where(scales > 0, 1.0 / np.where(scales > 0, scales, 1.0), 0.0)


def _quant_tensor_scale(x):
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max()
    s = amax / 448.0 if amax > 0 else 0.0
    codes = _e4m3(x / s) if s > 0 else np.zeros_like(x)
    return codes, np.full(x.shape[:-1], s)


_qproj = O.q_projection


def _qproj_whole_row_norm(qlat, wq, n_heads, head_dim, norm=True, eps=0.0, norm_w=None, store_bf16=False):
    y = _qproj(qlat, wq, n_heads, head_dim, norm=False)
    B, T = y.shape[:2]
    f = y.reshape(B, T, -1)
    f = f / np.sqrt(np.mean(f * f, axis=-1, keepdims=True) + eps)
    return f.reshape(y.shape)


def _qproj_transposed_weight(qlat, wq, n_heads, head_dim, norm=True, eps=0.0, norm_w=None, store_bf16=False):
    # the [r][H*D] weight read as if it were stored [H*D][r]
    r = np.asarray(qlat).shape[-1]
    w = np.asarray(wq).reshape(n_heads * head_dim, r).T
    return _qproj(qlat, w, n_heads, head_dim, norm, eps, norm_w, store_bf16)


_klt = O.indexer_kl_target


def _kl_sum_before_normalising(q, kv, ent, idx, sink, inv_freq, ratio, window, iscore=None, scale=None,
                               rows=None, rows_only=False):
    # heads summed as raw exponentials (one shared shift), normalised once
    q = np.asarray(q, dtype=np.float64)
    B, S, H, D = q.shape
    sc = D ** -0.5
    rows_ = np.arange(S) if rows is None else np.asarray(rows)
    out = _klt(q, kv, ent, idx, sink, inv_freq, ratio, window, iscore, scale, rows, rows_only)
    for b in range(B):
        for i, t in enumerate(rows_):
            slots = np.nonzero(np.asarray(idx)[b, t] >= 0)[0]
            if not len(slots):
                continue
            keys = O.attention_keys(0, 0, kv[b:b + 1], ent[b:b + 1], np.asarray(idx)[b:b + 1, t:t + 1], inv_freq,
                                    ratio, window, t=int(t))
            lg = sc * (O.rope_rotate(q[b, t], int(t), inv_freq) @ keys.T)
            e = np.exp(lg - lg.max()).sum(axis=0)[:len(slots)]
            out["target"][b, i, slots] = e / e.sum()
    return out


def _kl_entries_only(q, kv, ent, idx, sink, inv_freq, ratio, window, iscore=None, scale=None,
                     rows=None, rows_only=False):
    # per-head softmax over the selected entries alone (window, sink dropped)
    return _klt(q, kv, ent, idx, None, inv_freq, ratio, 0, iscore, scale, rows, rows_only)


def _kl_gradient_sign(q, kv, ent, idx, sink, inv_freq, ratio, window, iscore=None, scale=None,
                      rows=None, rows_only=False):
    out = _klt(q, kv, ent, idx, sink, inv_freq, ratio, window, iscore, scale, rows, rows_only)
    if out["dscore"] is not None:
        out["dscore"] = -out["dscore"]
    return out


MUTATIONS = [
    ("rope_rotate", _flip_sign, P.test_rope_is_complex_multiplication),
    ("sparse_mqa", _inflated_scale, P.test_softmax_scale_is_head_dim_power),
    ("topk_select", _ties_high, P.test_topk_matches_brute_force_sort),
    ("pooling_weights", _no_ape, P.test_ape_row_order_is_chronological),
    ("window_range", _window_off_by_one, P.test_hca_equals_dense_masked_sdpa),
    ("hadamard_matrix", _unnormalised_hadamard, P.test_indexer_scores_invariant_under_hadamard),
    ("compress", _rotate_at_entry_index, P.test_constant_score_gives_mean_of_members),
    ("round_to_e4m3", _e4m3_two_mantissa_bits, F.test_e4m3_code_points_and_range),
    ("round_to_e4m3", _e4m3_half_up, F.test_e4m3_matches_library_cast_in_range),
    ("round_to_e4m3", _e4m3_no_saturation, F.test_e4m3_saturates),
    ("quantize_e4m3_rows", _quant_inverted_scale, F.test_quantizer_error_within_half_spacing),
    ("quantize_e4m3_rows", _quant_tensor_scale, F.test_quantizer_row_maximum_lands_on_448),
    ("q_projection", _qproj_whole_row_norm, P.test_q_projection_heads_have_unit_rms_and_ignore_scale),
    ("q_projection", _qproj_transposed_weight, P.test_q_projection_matches_explicit_sums),
    ("indexer_kl_target", _kl_sum_before_normalising, KL.test_two_heads_without_window),
    ("indexer_kl_target", _kl_entries_only, KL.test_two_heads_with_window_mass),
    ("indexer_kl_target", _kl_gradient_sign, KL.test_loss_gradient_matches_central_differences),
]


@pytest.mark.parametrize("name,mutant,pin", MUTATIONS, ids=["%s-%s" % (m[0], m[1].__name__) for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, mutant, pin):
    monkeypatch.setattr(O, name, mutant)
    with pytest.raises(AssertionError):
        pin()
