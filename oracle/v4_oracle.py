"""CPU oracle for the DeepSeek-V4-Flash compressed attention forward, its query
and output projections, the gradient of its attention step and the indexer's
distillation target.

TEST INFRASTRUCTURE ONLY. This module is the slow, plain, float64 statement of
what the attention path computes. Only the tests, ``__graft_entry__.smoke()``
and the CPU-baseline / reference leg of ``bench.py`` may import it. The CUDA
library never calls it and shares no code with it.

Sources (the three pages the method is taken from):
  [PR]   Primus PR #930 "fix(deepseek-v4): correct V4-Flash attention math, wire
         the MoE balance loss", Part 1 items 1-6 and 8.
  [BLOG] "Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs with
         Primus", sections "The DeepSeek-V4-Flash architecture", "Three attention
         types, interleaved", "Kernel fusions", "Attention kernels for the three
         layer types".

Every floating-point step runs in float64.  Where the CUDA path stores a bf16
tensor between steps (pooled entries, indexer keys, prepared indexer queries,
the attention output), the oracle rounds to bf16 (nearest, ties to even) at the
same point when ``store_bf16`` is set.

Readings of points the pages leave open (the plainest reading consistent with
the rest of the pages):
  * pooling scores are per channel (a per-token scalar score is the special
    case of a score that is constant across channels);
  * a group member that does not exist (the previous group of entry 0) is left
    out of the softmax;
  * ``ape`` rows are chronological: with overlap the first ``ratio`` rows belong
    to the previous group, the last ``ratio`` rows to the entry's own tokens;
    projection half 0 carries the own tokens, half 1 the previous ones;
  * entry s covers tokens [r*s, r*s + r) and is visible to query t iff
    r*s + r - 1 <= t, i.e. s < (t + 1) // r; a trailing partial group is not an
    entry;
  * each pooled entry is RMS-normalised (weight g) before its rotation;
  * RoPE acts on interleaved pairs of the last R dims with the usual
    complex-multiply sign; de-rotation is rotation by the negated position;
  * the sliding window of query t is tokens [max(0, t - W + 1), t]
    (W = -1: all tokens <= t); window tokens and selected entries are separate
    keys (no de-duplication);
  * the indexer temperature (Hi * Di) ** -0.5 multiplies the per-head weights;
  * top-k keeps the min(K, n_vis) best entries, equal scores going to the
    lower index; short rows are padded with -1;
  * the optional attention sink is one extra logit per head that enters the
    softmax denominator only;
  * the attention backward is the exact gradient of this forward (the pages
    give its kernels, not its formulas): entry gradients are w.r.t. the stored
    rotated entries, window gradients w.r.t. the un-rotated latent;
  * the opt-in E4M3 indexer scales every query-head row and every key row by
    its absolute maximum (the pages name the format, not the scaling), and
    takes the quantisation decision in float32 as the kernel does;
  * the indexer distillation target sums the heads' attention probabilities
    (each normalised over all of its keys, window and sink included) on the
    selected entries and renormalises the sum over the selection slots.
"""
from __future__ import annotations

import math

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# Storage rounding
# ---------------------------------------------------------------------------
def round_to_bf16(x):
    """Round to the nearest bfloat16 value (ties to even); result kept in float64.

    bfloat16 keeps 8 significant bits.  With x = m * 2**e and 0.5 <= |m| < 1,
    the representable neighbours are multiples of 2**(e - 8); numpy's ``rint``
    rounds halfway cases to even.  Subnormal and overflowing values never occur
    on this path and are not treated specially.
    """
    x = np.asarray(x, dtype=F64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def maybe_bf16(x, store_bf16):
    return round_to_bf16(x) if store_bf16 else np.asarray(x, dtype=F64)


# ---------------------------------------------------------------------------
# RoPE tables and rotation  ([PR] items 2 and 8; [BLOG] "Kernel fusions",
# row "Interleaved partial RoPE")
# ---------------------------------------------------------------------------
def make_inv_freq(theta, rope_dim, yarn_factor=1.0, original_len=0,
                  beta_fast=32.0, beta_slow=1.0):
    """Inverse frequencies of the rotated pairs, returned as float32.

    Base table: theta ** (-2j / rope_dim) for pair j.  [PR] item 8 pairs the
    compressed base (40000 for Flash) with a YaRN factor (16) acting on this
    table.  YaRN's "NTK-by-parts" rule (Peng et al. 2023, section 3.2) is used:
    pair j has wavelength 2*pi / f_j; with ratio r_j = original_len / wavelength,
    the ramp gamma(r) is 0 below beta_slow, 1 above beta_fast and linear in
    between, and the new frequency is (1 - gamma) * f_j / s + gamma * f_j.
    Interpolation applies only when yarn_factor > 1 and original_len > 0 (the
    PR notes that the released model, with original_seq_len = 0, runs it off).
    """
    j = np.arange(rope_dim // 2, dtype=F64)
    f = np.power(F64(theta), -2.0 * j / F64(rope_dim))
    if yarn_factor > 1.0 and original_len > 0:
        wavelength = 2.0 * math.pi / f
        r = F64(original_len) / wavelength
        gamma = np.clip((r - beta_slow) / (beta_fast - beta_slow), 0.0, 1.0)
        f = (1.0 - gamma) * f / F64(yarn_factor) + gamma * f
    return f.astype(np.float32)


def yarn_attention_mscale(yarn_factor):
    """YaRN's attention temperature 0.1 * ln(s) + 1 (Peng et al. 2023).

    [PR] item 1: V4 must NOT multiply the softmax scale by this factor; the
    oracle keeps it only so a test can show the scale it would have inflated.
    """
    return 0.1 * math.log(yarn_factor) + 1.0 if yarn_factor > 1.0 else 1.0


def rope_rotate(x, pos, inv_freq):
    """Rotate interleaved pairs of the last R = 2 * len(inv_freq) dims.

    For pair j at channels (D-R+2j, D-R+2j+1) = (a, b) and angle
    phi = pos * inv_freq[j] (float64 from the float32 table):
        (a, b) -> (a cos phi - b sin phi, a sin phi + b cos phi).
    ``pos`` broadcasts against ``x.shape[:-1]``.
    """
    x = np.array(x, dtype=F64, copy=True)
    f = np.asarray(inv_freq, dtype=np.float32).astype(F64)
    R = 2 * f.shape[0]
    D = x.shape[-1]
    phi = np.asarray(pos, dtype=F64)[..., None] * f
    c, s = np.cos(phi), np.sin(phi)
    a = x[..., D - R::2].copy()
    b = x[..., D - R + 1::2].copy()
    x[..., D - R::2] = a * c - b * s
    x[..., D - R + 1::2] = a * s + b * c
    return x


def rope_derotate(x, pos, inv_freq):
    """[PR] item 3: rotation at the negated position (applied to the output)."""
    return rope_rotate(x, -np.asarray(pos, dtype=F64), inv_freq)


# ---------------------------------------------------------------------------
# Hadamard  ([PR] item 6e)
# ---------------------------------------------------------------------------
def hadamard_matrix(n):
    """Normalised Sylvester Hadamard matrix H_n / sqrt(n) (n a power of two)."""
    if n < 1 or (n & (n - 1)) != 0:
        raise ValueError("Hadamard size must be a power of two")
    h = np.ones((1, 1), dtype=F64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h / math.sqrt(n)


# ---------------------------------------------------------------------------
# Counting rules  ([BLOG] "Three attention types, interleaved")
# ---------------------------------------------------------------------------
def num_entries(seqlen, ratio):
    """Compressed entries of a sequence: one per complete group of ``ratio`` tokens."""
    return seqlen // ratio if ratio > 0 else 0


def n_visible(t, ratio):
    """Entries visible to query t: those whose last own token r*s + r - 1 <= t."""
    return (t + 1) // ratio if ratio > 0 else 0


def window_range(t, window):
    """Window tokens of query t as a half-open range [lo, t + 1)."""
    if window == 0:
        return t + 1, t + 1
    if window < 0:
        return 0, t + 1
    return max(0, t - window + 1), t + 1


def keys_read(t, ratio, window, topk):
    """Number of keys query t attends to (entries plus window tokens)."""
    nv = n_visible(t, ratio)
    ne = min(topk, nv) if topk > 0 else nv
    lo, hi = window_range(t, window)
    return ne + (hi - lo)


# ---------------------------------------------------------------------------
# Compressor  ([BLOG] "Three attention types, interleaved": shared learned
# pooling, CSA groups overlap; "Kernel fusions", row "Compressor pooling";
# [PR] items 2 and 6e)
# ---------------------------------------------------------------------------
def group_members(s, ratio, overlap):
    """(token, projection half, ape row) triples pooled into entry s."""
    members = []
    if overlap and s >= 1:
        for i in range(ratio):
            members.append((ratio * (s - 1) + i, 1, i))
    for i in range(ratio):
        members.append((ratio * s + i, 0, overlap * ratio + i))
    return members


def pooling_weights(cscore, ape, s, ratio, overlap):
    """Softmax over the group members of score + ape, per channel.

    cscore [B, S, 1+overlap, d]; returns (members, weights [B, G', d]).
    """
    members = group_members(s, ratio, overlap)
    lam = np.stack([cscore[:, j, half, :].astype(F64) + ape[row, :].astype(F64)
                    for (j, half, row) in members], axis=1)
    lam = lam - lam.max(axis=1, keepdims=True)
    e = np.exp(lam)
    return members, e / e.sum(axis=1, keepdims=True)


def compress(ckv, cscore, ape, norm_weight, inv_freq, ratio, overlap, eps,
             hadamard=False, store_bf16=False):
    """Pool the latent into compressed entries.

    ckv, cscore: [B, S, 1+overlap, d]; ape: [(1+overlap)*ratio, d] float32;
    norm_weight: [d] or None (ones).  Returns entries [B, N, d], N = S // ratio.
    Steps per entry s: pooled = sum_m softmax_m(score + ape) * ckv_m;
    e = pooled / sqrt(mean(pooled^2) + eps) * g; e = rot(e, ratio * s);
    indexer keys additionally take e = H e with the normalised Hadamard H.
    """
    ckv = np.asarray(ckv, dtype=F64)
    cscore = np.asarray(cscore, dtype=F64)
    B, S, P, d = ckv.shape
    if P != 1 + overlap:
        raise ValueError("ckv must carry 1 + overlap projection halves")
    N = num_entries(S, ratio)
    g = np.ones(d, dtype=F64) if norm_weight is None else np.asarray(norm_weight, dtype=F64)
    out = np.zeros((B, N, d), dtype=F64)
    for s in range(N):
        members, wts = pooling_weights(cscore, ape, s, ratio, overlap)
        vals = np.stack([ckv[:, j, half, :] for (j, half, _) in members], axis=1)
        out[:, s, :] = (wts * vals).sum(axis=1)
    rms = np.sqrt((out * out).mean(axis=-1, keepdims=True) + F64(eps))
    out = out / rms * g
    out = rope_rotate(out, (ratio * np.arange(N))[None, :], inv_freq)
    if hadamard:
        out = out @ hadamard_matrix(d).T
    return maybe_bf16(out, store_bf16)


# ---------------------------------------------------------------------------
# Lightning indexer  ([PR] items 4, 6a, 6e; [BLOG] "Kernel fusions", row
# "Indexer scoring tail"; "Three attention types": keep the best 512)
# ---------------------------------------------------------------------------
def indexer_scale(idx_heads, idx_dim):
    """[PR] item 6a: per-head weights scaled by Hi^-1/2 * Di^-1/2."""
    return 1.0 / math.sqrt(idx_heads) / math.sqrt(idx_dim)


def indexer_query_prep(iq, inv_freq, store_bf16=False, positions=None):
    """Queries rotated at their own positions t, then the normalised Hadamard.

    iq: [B, T, Hi, Di] -> same shape; row i sits at position positions[i]
    (default: positions 0..T-1).
    """
    iq = np.asarray(iq, dtype=F64)
    pos = np.arange(iq.shape[1]) if positions is None else np.asarray(positions)
    x = rope_rotate(iq, pos[None, :, None], inv_freq)
    x = x @ hadamard_matrix(iq.shape[-1]).T
    return maybe_bf16(x, store_bf16)


def indexer_scores(iq_prep, ikey, w, ratio, rows=None, rows_only=False):
    """I[b, t, s] = sum_h w[b,t,h] * (Hi*Di)^-1/2 * max(0, q~[b,t,h] . k[b,s]).

    Defined for s < n_visible(t); other entries are -inf.  ``rows`` selects the
    query positions (default: all); with ``rows_only`` the query and weight
    arrays hold just those rows, in order.  Returns [B, len(rows), N].
    """
    iq_prep = np.asarray(iq_prep, dtype=F64)
    ikey = np.asarray(ikey, dtype=F64)
    w = np.asarray(w, dtype=F64)
    B, S, Hi, Di = iq_prep.shape
    N = ikey.shape[1]
    rows = np.arange(S) if rows is None else np.asarray(rows)
    c = indexer_scale(Hi, Di)
    out = np.full((B, len(rows), N), -np.inf, dtype=F64)
    for b in range(B):
        for i, t in enumerate(rows):
            nv = min(n_visible(int(t), ratio), N)
            if nv == 0:
                continue
            r = i if rows_only else t
            dots = iq_prep[b, r] @ ikey[b, :nv].T          # [Hi, nv]
            out[b, i, :nv] = (w[b, r] * c) @ np.maximum(dots, 0.0)
    return out


def topk_select(score_row, nvis, k):
    """Best min(k, nvis) entries of one row; ties go to the lower index.

    Returns (indices [k] int32 padded with -1, scores [k] padded with -inf),
    ordered by decreasing score.
    """
    nvis = int(nvis)
    idx = np.full(k, -1, dtype=np.int32)
    val = np.full(k, -np.inf, dtype=F64)
    if nvis <= 0 or k <= 0:
        return idx, val
    s = np.arange(nvis)
    order = np.lexsort((s, -np.asarray(score_row[:nvis], dtype=F64)))
    take = order[:min(k, nvis)]
    idx[:len(take)] = take
    val[:len(take)] = score_row[take]
    return idx, val


def indexer_topk(iq, ikey, w, inv_freq, ratio, k, store_bf16=False, rows=None,
                 prepared=False, rows_only=False):
    """Indexer from un-rotated queries (or prepared ones) to top-k index sets.

    With ``rows_only`` the iq and w arrays hold just the listed rows.
    Returns dict(idx [B,T,k] int32, iscore [B,T,k], scores [B,T,N]).
    """
    S = np.asarray(iq).shape[1]
    rows_ = np.arange(S) if rows is None else np.asarray(rows)
    if not rows_only and rows is not None:
        iq = np.asarray(iq)[:, rows_]
        w = np.asarray(w)[:, rows_]
    qp = np.asarray(iq, dtype=F64) if prepared else indexer_query_prep(iq, inv_freq, store_bf16,
                                                                       positions=rows_)
    sc = indexer_scores(qp, ikey, w, ratio, rows_, rows_only=True)
    B, T, N = sc.shape
    idx = np.full((B, T, k), -1, dtype=np.int32)
    isc = np.full((B, T, k), -np.inf, dtype=F64)
    for b in range(B):
        for i, t in enumerate(rows_):
            idx[b, i], isc[b, i] = topk_select(sc[b, i], min(n_visible(int(t), ratio), N), k)
    return {"idx": idx, "iscore": isc, "scores": sc}


# ---------------------------------------------------------------------------
# Opt-in E4M3 indexer QK  ([PR] item 4: the indexer QK stays in high
# precision by default, FP8 only behind its own switch, because quantisation
# error changes the selection; [BLOG] closing section: an E4M3 path for the
# indexer QK ships)
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0


def round_to_e4m3(x):
    """Nearest E4M3 ("FN": no infinities) value, ties to even, saturating.

    E4M3 has 1 sign, 4 exponent (bias 7) and 3 mantissa bits.  Normal values
    are (1 + m/8) * 2**(e-7) for e = 1..15, except that e = 15 with m = 7 is
    NaN, so the largest finite value is 1.75 * 2**8 = 448; subnormals are
    m/8 * 2**-6.  Hence for |x| >= 2**-6 the spacing is 2**(floor(log2|x|) - 3)
    and below 2**-6 it is 2**-9.  Rounding to the nearest multiple of the
    spacing with numpy's ``rint`` sends halfway cases to the even significand;
    magnitudes beyond 448 saturate to 448 (the "satfinite" conversion).
    Result kept in float64.
    """
    x = np.asarray(x, dtype=F64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))      # a = m * 2**ex, 0.5 <= m < 1
    e = np.maximum(ex - 1, -6)                      # floor(log2 a), clamped to the subnormal range
    q = np.ldexp(1.0, e - 3)
    r = np.minimum(np.rint(a / q) * q, E4M3_MAX)
    return np.copysign(r, x)


def quantize_e4m3_rows(x):
    """Per-row absolute-maximum scaling of x [..., dim] to E4M3.

    The plainest reading of an E4M3 QK (the pages name the format, not the
    scaling): each row (one query head, one key) gets scale = amax / 448 and
    code = e4m3(x * (448 / amax)), so that x ~= code * scale.  The code is an
    integer-like decision taken in float32 as the kernel takes it: amax is
    exact (x holds bf16 values), 448 / amax and amax / 448 are float32
    divisions and x * inv a float32 product, each rounded to nearest.  An
    all-zero row has scale 0 and zero codes.
    Returns (codes [..., dim] float64 values of E4M3 numbers, scales [...]).
    """
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    pos = amax > 0
    one = np.float32(E4M3_MAX)
    safe = np.where(pos, amax, np.float32(1.0)).astype(np.float32)
    inv = np.where(pos, one / safe, np.float32(0.0)).astype(np.float32)
    scale = np.where(pos, safe / one, np.float32(0.0)).astype(np.float32)
    prod = (x32 * inv[..., None]).astype(np.float32)
    return round_to_e4m3(prod.astype(F64)), scale.astype(F64)


def indexer_scores_e4m3(q_codes, q_scales, k_codes, k_scales, w, ratio, rows=None, rows_only=False):
    """Indexer scores of quantised operands: q~[t,h] = q_codes * q_scales[t,h]
    and k[s] = k_codes * k_scales[s] dequantised exactly (float64), then the
    scores of ``indexer_scores``.  Same arguments and result shape."""
    qd = np.asarray(q_codes, dtype=F64) * np.asarray(q_scales, dtype=F64)[..., None]
    kd = np.asarray(k_codes, dtype=F64) * np.asarray(k_scales, dtype=F64)[..., None]
    return indexer_scores(qd, kd, w, ratio, rows, rows_only)


def indexer_topk_e4m3(q_codes, q_scales, k_codes, k_scales, w, ratio, k, rows=None, rows_only=False):
    """Top-k selection of the E4M3 scores (same rules as ``indexer_topk``)."""
    S = np.asarray(q_codes).shape[1]
    rows_ = np.arange(S) if rows is None else np.asarray(rows)
    sc = indexer_scores_e4m3(q_codes, q_scales, k_codes, k_scales, w, ratio, rows_, rows_only)
    B, T, N = sc.shape
    idx = np.full((B, T, k), -1, dtype=np.int32)
    isc = np.full((B, T, k), -np.inf, dtype=F64)
    for b in range(B):
        for i, t in enumerate(rows_):
            idx[b, i], isc[b, i] = topk_select(sc[b, i], min(n_visible(int(t), ratio), N), k)
    return {"idx": idx, "iscore": isc, "scores": sc}


# ---------------------------------------------------------------------------
# Sparse / dense multi-query attention  ([BLOG] "The DeepSeek-V4-Flash
# architecture": 64 heads share one 512-d latent that is both key and value;
# "Three attention types": selected entries plus a 128-token window; "Kernel
# fusions", row "SWA / CSA / HCA attention": window and sink in one softmax;
# [PR] item 1: scale head_dim ** -0.5; item 3: de-rotate the output at -t)
# ---------------------------------------------------------------------------
def attention_keys(b, i, kv, ent, idx, inv_freq, ratio, window, t=None):
    """Keys (= values) of query t: the chosen entries, then the window tokens.

    idx row i of batch b lists query t's selection (t defaults to i).
    """
    t = i if t is None else t
    parts = []
    if ratio > 0 and ent is not None:
        nv = min(n_visible(t, ratio), ent.shape[1])
        if idx is not None:
            sel = np.asarray(idx[b, i])
            sel = sel[sel >= 0]
            if np.any(sel >= nv):
                raise ValueError("selected entry is not causally visible")
        else:
            sel = np.arange(nv)
        parts.append(np.asarray(ent[b, sel], dtype=F64))
    lo, hi = window_range(t, window)
    if hi > lo:
        u = np.arange(lo, hi)
        parts.append(rope_rotate(np.asarray(kv[b, lo:hi], dtype=F64), u, inv_freq))
    if not parts:
        return np.zeros((0, kv.shape[-1]), dtype=F64)
    return np.concatenate(parts, axis=0)


def sparse_mqa(q, kv, ent, idx, sink, inv_freq, ratio, window, scale=None,
               store_bf16=False, rows=None, rows_only=False):
    """Attention of every head of query t over its keys, de-rotated at -t.

    q [B,S,H,D] (un-rotated), kv [B,S,D] (un-rotated window latent),
    ent [B,N,D] (rotated entries) or None, idx [B,S,K] or None (all visible),
    sink [H] or None.  Returns (o [B,T,H,D], lse [B,T,H]) for the ``rows``.
    logits = scale * rot(q_h, t) . key; m = max(logits, sink);
    o = sum_j exp(l_j - m) key_j / (sum_j exp(l_j - m) + exp(sink - m)).
    An empty key set without a sink gives o = 0, lse = -inf.  With
    ``rows_only`` q and idx hold just the listed rows, in order.
    """
    q = np.asarray(q, dtype=F64)
    B, S, H, D = q.shape
    scale = D ** -0.5 if (scale is None or scale <= 0) else scale
    rows = np.arange(S) if rows is None else np.asarray(rows)
    o = np.zeros((B, len(rows), H, D), dtype=F64)
    lse = np.full((B, len(rows), H), -np.inf, dtype=F64)
    z = None if sink is None else np.asarray(sink, dtype=F64)
    for b in range(B):
        for i, t in enumerate(rows):
            t = int(t)
            r = i if rows_only else t
            sel = None if idx is None else np.asarray(idx)[b:b + 1, r:r + 1]
            keys = attention_keys(0, 0, kv[b:b + 1], None if ent is None else ent[b:b + 1], sel,
                                  inv_freq, ratio, window, t=t)
            qr = rope_rotate(q[b, r], t, inv_freq)               # [H, D]
            logits = scale * (qr @ keys.T)                       # [H, nk]
            if keys.shape[0] == 0 and z is None:
                continue
            m = logits.max(axis=1) if keys.shape[0] else np.full(H, -np.inf)
            if z is not None:
                m = np.maximum(m, z)
            e = np.exp(logits - m[:, None])
            den = e.sum(axis=1)
            if z is not None:
                den = den + np.exp(z - m)
            out = (e @ keys) / den[:, None]
            o[b, i] = rope_derotate(out, t, inv_freq)
            lse[b, i] = m + np.log(den)
    return maybe_bf16(o, store_bf16), lse


# ---------------------------------------------------------------------------
# Sparse indexer distillation target  ([PR] item 5: KL(attention || indexer)
# over the selected entries, the sparse top-k variant kept in [B, S, K];
# item 11: the target branch is detached, head-summed inside the loop)
# ---------------------------------------------------------------------------
def indexer_kl_target(q, kv, ent, idx, sink, inv_freq, ratio, window, iscore=None, scale=None,
                      rows=None, rows_only=False):
    """Target distribution of the indexer and the KL loss, per query t.

    A_h = the main attention's probabilities of head h over all of t's keys
    (selected entries, window tokens, sink in the denominator), as in
    ``sparse_mqa``.  The target over t's selection slots is the head sum of
    A on the selected entries, L1-normalised over the slots:
        p[t, k] = sum_h A_h[idx[t,k]] / sum_k' sum_h A_h[idx[t,k']]
    (0 on padding slots, and everywhere when the entries carry no mass).
    With ``iscore`` (the indexer's scores of the slots) the indexer's
    distribution is qd = softmax over the valid slots, the loss is
    KL(p || qd) = sum_k p (log p - log qd) (0 log 0 = 0) and its gradient
    with respect to iscore is qd - p.
    Returns dict(target [B,T,K], loss [B,T] or None, dscore [B,T,K] or None).
    """
    q = np.asarray(q, dtype=F64)
    B, S, H, D = q.shape
    scale = D ** -0.5 if (scale is None or scale <= 0) else scale
    rows = np.arange(S) if rows is None else np.asarray(rows)
    idx = np.asarray(idx)
    K = idx.shape[-1]
    z = None if sink is None else np.asarray(sink, dtype=F64)
    target = np.zeros((B, len(rows), K), dtype=F64)
    loss = np.zeros((B, len(rows)), dtype=F64) if iscore is not None else None
    dscore = np.zeros((B, len(rows), K), dtype=F64) if iscore is not None else None
    for b in range(B):
        for i, t in enumerate(rows):
            t = int(t)
            r = i if rows_only else t
            slots = np.nonzero(idx[b, r] >= 0)[0]
            if len(slots) == 0:
                continue
            keys = attention_keys(0, 0, kv[b:b + 1], ent[b:b + 1], idx[b:b + 1, r:r + 1], inv_freq,
                                  ratio, window, t=t)
            qr = rope_rotate(q[b, r], t, inv_freq)
            logits = scale * (qr @ keys.T)                      # [H, nk]; entries first, in slot order
            m = logits.max(axis=1)
            if z is not None:
                m = np.maximum(m, z)
            e = np.exp(logits - m[:, None])
            den = e.sum(axis=1)
            if z is not None:
                den = den + np.exp(z - m)
            A = e / den[:, None]
            raw = A[:, :len(slots)].sum(axis=0)
            tot = raw.sum()
            pk = raw / tot if tot > 0 else np.zeros_like(raw)
            target[b, i, slots] = pk
            if iscore is not None:
                sc = np.asarray(iscore, dtype=F64)[b, r, slots]
                lq = sc - sc.max()
                lq = lq - np.log(np.exp(lq).sum())
                qd = np.exp(lq)
                nz = pk > 0
                loss[b, i] = float(np.sum(pk[nz] * (np.log(pk[nz]) - lq[nz])))
                dscore[b, i, slots] = qd - pk
    return {"target": target, "loss": loss, "dscore": dscore}


# ---------------------------------------------------------------------------
# Attention backward  ([BLOG] "Attention kernels for the three layer types",
# backward: the gradient of the same forward, split there into dQ, a
# head-dimension contraction ("interm") and the delta rowsum(O * dO))
# ---------------------------------------------------------------------------
def sparse_mqa_bwd(q, kv, ent, idx, sink, inv_freq, ratio, window, dout, scale=None, rows=None):
    """Exact gradients of L = sum(dout * o) for o = sparse_mqa(...).

    Written out by the chain rule for one query t with keys k_j (chosen
    entries, then window tokens rotated at their positions u) and
    qr_h = rot(q_h, t):
        p_hj   = exp(scale qr_h . k_j - lse_h)      (the sink takes the rest)
        g_h    = rot(dout_h, t)                     (o = rot(o', -t), o' = sum_j p_hj k_j)
        delta_h = g_h . o'_h  (= dout_h . o_h, rotation is orthogonal)
        ds_hj  = p_hj (g_h . k_j - delta_h)         (gradient of the logit)
        dq_h   = rot(scale sum_j ds_hj k_j, -t)
        dk_j   = scale sum_h ds_hj qr_h + sum_h p_hj g_h   (key = value)
        dsink_h = -p_sink,h delta_h,  p_sink,h = exp(sink_h - lse_h)
    Entry gradients are taken w.r.t. the stored (rotated) entries; window
    gradients w.r.t. the un-rotated latent kv, i.e. rot(dk_u, -u).

    q, dout [B,S,H,D] and idx [B,S,K] are indexed by position t.
    Returns dq [B,T,H,D] for the ``rows`` (all by default), dkv [B,S,D],
    dent [B,N,D] (None without entries) and dsink [H] (None without sink);
    dkv, dent and dsink hold the contributions of the listed rows only.
    """
    q = np.asarray(q, dtype=F64)
    dout = np.asarray(dout, dtype=F64)
    kv = np.asarray(kv, dtype=F64)
    B, S, H, D = q.shape
    scale = D ** -0.5 if (scale is None or scale <= 0) else scale
    rows = np.arange(S) if rows is None else np.asarray(rows)
    have_ent = ratio > 0 and ent is not None
    entf = np.asarray(ent, dtype=F64) if have_ent else None
    z = None if sink is None else np.asarray(sink, dtype=F64)
    dq = np.zeros((B, len(rows), H, D), dtype=F64)
    dkv = np.zeros((B, S, D), dtype=F64)
    dent = np.zeros_like(entf) if have_ent else None
    dsink = np.zeros(H, dtype=F64) if z is not None else None
    for b in range(B):
        for i, t in enumerate(rows):
            t = int(t)
            sel = np.zeros(0, dtype=np.int64)
            if have_ent:
                nv = min(n_visible(t, ratio), entf.shape[1])
                if idx is not None:
                    sel = np.asarray(idx[b, t])
                    sel = sel[sel >= 0].astype(np.int64)
                    if np.any(sel >= nv):
                        raise ValueError("selected entry is not causally visible")
                else:
                    sel = np.arange(nv)
            lo, hi = window_range(t, window)
            u = np.arange(lo, hi)
            keys = np.concatenate([entf[b, sel] if have_ent else np.zeros((0, D)),
                                   rope_rotate(kv[b, lo:hi], u, inv_freq)], axis=0)
            if keys.shape[0] == 0:
                continue                                   # o = 0 whatever the inputs
            qr = rope_rotate(q[b, t], t, inv_freq)         # [H, D]
            logits = scale * (qr @ keys.T)                 # [H, nk]
            m = logits.max(axis=1)
            if z is not None:
                m = np.maximum(m, z)
            e = np.exp(logits - m[:, None])
            den = e.sum(axis=1) + (np.exp(z - m) if z is not None else 0.0)
            p = e / den[:, None]
            o_rot = p @ keys                               # [H, D], before de-rotation
            g = rope_rotate(dout[b, t], t, inv_freq)       # gradient of o_rot
            delta = (g * o_rot).sum(axis=1)
            ds = p * (g @ keys.T - delta[:, None])
            dq[b, i] = rope_derotate(scale * (ds @ keys), t, inv_freq)
            dk = scale * (ds.T @ qr) + p.T @ g             # [nk, D]
            ns = sel.shape[0]
            if ns:
                np.add.at(dent[b], sel, dk[:ns])
            if hi > lo:
                dkv[b, lo:hi] += rope_derotate(dk[ns:], u, inv_freq)
            if z is not None:
                dsink -= np.exp(z - m) / den * delta
    return dq, dkv, dent, dsink


# ---------------------------------------------------------------------------
# Grouped low-rank output projection  ([BLOG] "The DeepSeek-V4-Flash
# architecture": 8 groups, each through a 1024-d bottleneck)
# ---------------------------------------------------------------------------
def grouped_wo_a(o, wo_a, store_bf16=False):
    """y[b,t,g,:] = concat_{h in group g} o[b,t,h,:] @ wo_a[g].

    o [B,T,H,D]; wo_a [G, (H/G)*D, rank]; returns [B, T, G*rank].
    Group g holds heads g*H/G .. (g+1)*H/G - 1, concatenated along D.
    """
    o = np.asarray(o, dtype=F64)
    B, T, H, D = o.shape
    G, gin, rank = wo_a.shape
    x = o.reshape(B * T, G, gin)
    w = np.asarray(wo_a, dtype=F64)
    y = np.stack([x[:, g, :] @ w[g] for g in range(G)], axis=1)      # [B*T, G, rank]
    return maybe_bf16(y.reshape(B, T, G * rank), store_bf16)


# ---------------------------------------------------------------------------
# Query projections  ([BLOG] "The DeepSeek-V4-Flash architecture": queries
# arrive through a low-rank path of rank 1024 that the indexer shares)
# ---------------------------------------------------------------------------
def q_projection(qlat, wq, n_heads, head_dim, norm=True, eps=0.0, norm_w=None, store_bf16=False):
    """Attention queries from the shared rank-r latent.

    qlat [B,T,r], wq [r, H*D]; y = qlat @ wq viewed as [B,T,H,D].  With
    ``norm`` every head is RMS-normalised over its D dims (the reading the
    benchmark inputs use: unit-RMS heads), y / sqrt(mean(y^2) + eps) * g,
    g = norm_w [D] or ones.  Returns [B,T,H,D].
    """
    qlat = np.asarray(qlat, dtype=F64)
    B, T, r = qlat.shape
    y = (qlat.reshape(B * T, r) @ np.asarray(wq, dtype=F64)).reshape(B, T, n_heads, head_dim)
    if norm:
        y = y / np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + eps)
        if norm_w is not None:
            y = y * np.asarray(norm_w, dtype=F64)
    return maybe_bf16(y, store_bf16)


def indexer_q_projection(qlat, wiq, idx_heads, idx_dim, store_bf16=False):
    """Indexer queries from the same latent: qlat @ wiq viewed as [B,T,Hi,Di]."""
    qlat = np.asarray(qlat, dtype=F64)
    B, T, r = qlat.shape
    y = (qlat.reshape(B * T, r) @ np.asarray(wiq, dtype=F64)).reshape(B, T, idx_heads, idx_dim)
    return maybe_bf16(y, store_bf16)


# ---------------------------------------------------------------------------
# One attention layer
# ---------------------------------------------------------------------------
def attn_layer(cfg, x, rows=None):
    """Whole forward of one layer as the CUDA library composes it.

    cfg: dict with ratio, overlap, window, topk, rms_eps, store_bf16 and
    optionally softmax_scale.  x: dict of numpy inputs (q, kv, ckv, cscore, ape,
    norm_w, ickv, icscore, iape, inorm_w, iq, w, sink, inv_freq, wo_a).
    Returns dict with ent, ikey, idx, iscore, o, lse and (if wo_a) y.
    """
    r, ov, W, K = cfg["ratio"], cfg["overlap"], cfg["window"], cfg["topk"]
    bf = cfg.get("store_bf16", False)
    eps = cfg.get("rms_eps", 1e-6)
    res = {"ent": None, "ikey": None, "idx": None, "iscore": None}
    if r > 0:
        res["ent"] = compress(x["ckv"], x["cscore"], x["ape"], x.get("norm_w"),
                              x["inv_freq"], r, ov, eps, hadamard=False, store_bf16=bf)
        if K > 0:
            res["ikey"] = compress(x["ickv"], x["icscore"], x["iape"], x.get("inorm_w"),
                                   x["inv_freq"], r, ov, eps, hadamard=True, store_bf16=bf)
            sel = indexer_topk(x["iq"], res["ikey"], x["w"], x["inv_freq"], r, K,
                               store_bf16=bf, rows=rows)
            res["idx"], res["iscore"] = sel["idx"], sel["iscore"]
    idx_full = None
    if res["idx"] is not None:
        # sparse_mqa indexes idx by absolute position; scatter the sampled rows.
        B, S = x["q"].shape[:2]
        idx_full = np.full((B, S, K), -1, dtype=np.int32)
        rr = np.arange(S) if rows is None else np.asarray(rows)
        idx_full[:, rr] = res["idx"]
    o, lse = sparse_mqa(x["q"], x["kv"], res["ent"], idx_full, x.get("sink"),
                        x["inv_freq"], r, W, cfg.get("softmax_scale"),
                        store_bf16=bf, rows=rows)
    res["o"], res["lse"] = o, lse
    if x.get("wo_a") is not None:
        res["y"] = grouped_wo_a(o, x["wo_a"], store_bf16=bf)
    return res
