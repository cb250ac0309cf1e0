"""Pins of the oracle's sparse indexer distillation target (CPU only).

Hand-computed two-head cases fix that heads are normalised over all their
keys (window and sink included) before the head sum, and only then is the
sum renormalised over the selection; one head whose indexer scores equal its
logits gives a zero loss; the loss is non-negative and its stated gradient
matches central differences; the target is a distribution over the valid
slots and moves with them when the slots are permuted.
"""
import math

import numpy as np
import pytest

from oracle import v4_oracle as O


def _two_head_case(window):
    # D = 4, no rotated dims, ratio 1 (every token is an entry); query t = 2
    # selects entries 0 and 1; with window 1 its own token is a third key.
    D, S = 4, 3
    s = D ** -0.5
    ent = np.zeros((1, S, D))
    ent[0, 0, 0] = 1.0
    ent[0, 1, 1] = 1.0
    kv = np.zeros((1, S, D))
    kv[0, 2, 2] = 1.0
    q = np.zeros((1, S, 2, D))
    q[0, 2, 0, 0] = math.log(9.0) / s
    q[0, 2, 0, 2] = math.log(10.0) / s
    idx = np.full((1, S, 2), -1)
    idx[0, 2] = [0, 1]
    f = np.zeros(0, dtype=np.float32)
    return O.indexer_kl_target(q, kv, ent, idx, None, f, 1, window, rows=[2])["target"][0, 0]


def test_two_heads_without_window():
    # head 1: softmax(ln 9, 0) = (0.9, 0.1); head 2: (0.5, 0.5)
    np.testing.assert_allclose(_two_head_case(0), [0.7, 0.3], rtol=1e-12)


def test_two_heads_with_window_mass():
    # head 1 over (entry 0, entry 1, own token): (9, 1, 10) / 20; head 2: thirds
    raw = np.array([0.45 + 1 / 3, 0.05 + 1 / 3])
    np.testing.assert_allclose(_two_head_case(1), raw / raw.sum(), rtol=1e-12)


def _random_case(seed, H=3, D=16, R=4, S=40, r=2, K=6, W=3, sink=True):
    rng = np.random.default_rng(seed)
    N = S // r
    q = rng.normal(0, 1, (1, S, H, D))
    kv = rng.normal(0, 1, (1, S, D))
    ent = rng.normal(0, 1, (1, N, D))
    f = O.make_inv_freq(10000.0, R)
    idx = np.full((1, S, K), -1)
    for t in range(S):
        nv = min(O.n_visible(t, r), N)
        sel = rng.permutation(nv)[:K]
        slots = rng.permutation(K)[:len(sel)]
        idx[0, t, slots] = sel
    z = rng.normal(0, 1, H) if sink else None
    isc = rng.normal(0, 2, (1, S, K))
    return q, kv, ent, idx, z, f, r, W, isc


def test_one_head_scores_equal_to_logits_give_zero_loss():
    q, kv, ent, idx, _, f, r, _, _ = _random_case(1, H=1)
    S, K = idx.shape[1:]
    isc = np.zeros((1, S, K))
    D = q.shape[-1]
    for t in range(S):
        for k in range(K):
            e = idx[0, t, k]
            if e >= 0:
                isc[0, t, k] = D ** -0.5 * O.rope_rotate(q[0, t, 0], t, f) @ ent[0, e] + 3.0
    out = O.indexer_kl_target(q, kv, ent, idx, None, f, r, 0, iscore=isc)
    np.testing.assert_allclose(out["loss"], 0.0, atol=1e-12)
    np.testing.assert_allclose(out["dscore"], 0.0, atol=1e-12)


def test_target_is_a_distribution_over_valid_slots():
    q, kv, ent, idx, z, f, r, W, isc = _random_case(2)
    out = O.indexer_kl_target(q, kv, ent, idx, z, f, r, W, iscore=isc)
    p = out["target"][0]
    valid = idx[0] >= 0
    assert np.all(p[~valid] == 0) and np.all(p >= 0)
    rows = valid.any(axis=1)
    np.testing.assert_allclose(p[rows].sum(axis=1), 1.0, rtol=1e-12)
    assert np.all(out["loss"] >= -1e-12)
    np.testing.assert_allclose(out["dscore"][0][rows].sum(axis=1), 0.0, atol=1e-12)


def test_loss_gradient_matches_central_differences():
    q, kv, ent, idx, z, f, r, W, isc = _random_case(3)
    out = O.indexer_kl_target(q, kv, ent, idx, z, f, r, W, iscore=isc)
    rng = np.random.default_rng(4)
    h = 1e-6
    for _ in range(12):
        t = int(rng.integers(4, idx.shape[1]))
        ks = np.nonzero(idx[0, t] >= 0)[0]
        k = int(rng.choice(ks))
        a, b = isc.copy(), isc.copy()
        a[0, t, k] += h
        b[0, t, k] -= h
        la = O.indexer_kl_target(q, kv, ent, idx, z, f, r, W, iscore=a, rows=[t])["loss"][0, 0]
        lb = O.indexer_kl_target(q, kv, ent, idx, z, f, r, W, iscore=b, rows=[t])["loss"][0, 0]
        assert abs((la - lb) / (2 * h) - out["dscore"][0, t, k]) < 1e-6


def test_target_follows_permuted_slots():
    q, kv, ent, idx, z, f, r, W, _ = _random_case(5)
    p = O.indexer_kl_target(q, kv, ent, idx, z, f, r, W)["target"]
    perm = np.random.default_rng(6).permutation(idx.shape[-1])
    p2 = O.indexer_kl_target(q, kv, ent, idx[..., perm], z, f, r, W)["target"]
    np.testing.assert_allclose(p2, p[..., perm], rtol=1e-12, atol=1e-15)
