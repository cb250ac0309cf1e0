"""Shared test utilities: input staging, tolerance checks, oracle runners."""
import math

import numpy as np
import torch

import seeded_inputs as SI
from oracle import v4_oracle as O

U32 = 2.0 ** -24     # fp32 unit roundoff


def np64(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def assert_within_bf16_ulp(gpu, ref, ulps=1, frac_exact_min=None, row_terms=None):
    """Every element within `ulps` bf16 ulps of the oracle's bf16-rounded value,
    plus the fp32 forward-error allowance of the kernel's arithmetic.

    The kernels compute in fp32 and round once to bf16.  An output that comes
    out of a cancelling sum (the Hadamard, a rotation) carries an absolute fp32
    error proportional to the magnitude of the row, not of the result, so
    each element also gets row_terms * 2^-24 * max|row| (row = last axis).
    """
    g = np64(gpu)
    r = np.asarray(ref, dtype=np.float64)
    m, e = np.frexp(np.abs(r))
    ulp = np.ldexp(1.0, e - 8)
    ulp = np.where(r == 0, 2.0 ** -133, ulp)
    allow = ulps * ulp + 1e-30
    if row_terms is not None:
        allow = allow + row_terms * U32 * np.abs(r).max(axis=-1, keepdims=True)
    err = np.abs(g - r)
    bad = err > allow
    if bad.any():
        k = int(np.argmax((err / allow).ravel()))
        raise AssertionError("%d of %d elements beyond tolerance; worst: gpu %r oracle %r allow %r" % (
            bad.sum(), bad.size, g.ravel()[k], r.ravel()[k], allow.ravel()[k]))
    if frac_exact_min is not None:
        assert np.mean(g == r) >= frac_exact_min


def inv_freq_for(p):
    yarn = p.get("yarn", 1.0)
    return O.make_inv_freq(p["theta"], p["R"], yarn, SI.YARN_ORIGINAL_LEN if yarn > 1 else 0,
                           SI.YARN_BETA_FAST, SI.YARN_BETA_SLOW)


def to_dev(x, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def oracle_inputs(x, f):
    """numpy float64 views of the generator's tensors, for the oracle."""
    out = {k: np64(v) for k, v in x.items()}
    out["inv_freq"] = f
    return out


def topk_fp32_band(iqp, ikey, w, t, nvis, c):
    """Forward error bound of the fp32 score arithmetic for row t.

    |delta I| <= 4 * ((Di+2) u sum_h |w_h c| sum_c |q k| + (Hi+2) u sum_h |w_h c| |d_h|),
    maximised over the visible entries (u = 2^-24).
    """
    q = np.abs(iqp[t])                        # [Hi, Di]
    k = np.abs(ikey[:nvis])                   # [nv, Di]
    wa = np.abs(w[t]) * c                     # [Hi]
    absdot = q @ k.T                          # [Hi, nv]
    d = np.abs(iqp[t] @ ikey[:nvis].T)
    Hi, Di = iqp.shape[-2:]
    b = 4.0 * ((Di + 2) * U32 * (wa @ absdot) + (Hi + 2) * U32 * (wa @ d))
    return float(b.max()) if b.size else 0.0


def check_topk_rows(gpu_idx, scores, iqp, ikey, w, ratio, K, rows, c, detail=False):
    """Set-exact selection outside the tie band around the K-th score.

    gpu_idx [T, K] int; scores [T, N] oracle float64; iqp/ikey/w: the exact
    inputs (float64 numpy) of one batch.  The band is the larger of
    1e-6 * |I_K| (the tie rule of the selection's specification) and the
    forward-error bound of the fp32 score arithmetic.  Returns the number of
    in-band swaps (entries of the exact top-K the GPU left out); with
    ``detail`` also the number of swapped entries (left out or taken) whose
    exact score lies outside the strict 1e-6 * |I_K| band, i.e. swaps that
    only the fp32 error bound allows.
    """
    swaps = 0
    wide = 0
    for i, t in enumerate(rows):
        nv = min(O.n_visible(int(t), ratio), ikey.shape[0])
        g = gpu_idx[i]
        sel = g[g >= 0]
        assert len(sel) == min(K, nv), (t, len(sel), min(K, nv))
        assert len(set(sel.tolist())) == len(sel), "duplicate index in row %d" % t
        assert np.all(sel < nv), "invisible entry selected in row %d" % t
        if nv <= K:
            assert set(sel.tolist()) == set(range(nv))
            continue
        row = scores[i, :nv]
        kth = np.sort(row)[::-1][K - 1]
        band = max(1e-6 * abs(kth), topk_fp32_band(iqp, ikey, w, int(t), nv, c))
        must_in = set(np.nonzero(row > kth + band)[0].tolist())
        must_out = set(np.nonzero(row < kth - band)[0].tolist())
        s = set(sel.tolist())
        assert must_in <= s, "row %d misses %s" % (t, sorted(must_in - s)[:5])
        assert not (s & must_out), "row %d takes %s" % (t, sorted(s & must_out)[:5])
        ref = set(O.topk_select(row, nv, K)[0].tolist())
        swaps += len(ref - s)
        strict = 1e-6 * abs(kth)
        wide += sum(1 for e in (ref ^ s) if abs(row[e] - kth) > strict)
    return (swaps, wide) if detail else swaps


def check_attention_rows(o, lse, ro, rl, tol=1e-2, lse_extra=0.0):
    """Attention outputs against the oracle: relative L2 over all rows,
    every row within 5 * tol, and lse within the bf16 operand error
    (plus lse_extra, broadcast over [B, S, H], for inputs scaled beyond
    unit size)."""
    assert rel_l2(o, ro) < tol
    B, S, H, D = o.shape
    num = np.linalg.norm((o - ro).reshape(B * S, -1), axis=1)
    den = np.linalg.norm(ro.reshape(B * S, -1), axis=1) + 1e-30
    assert np.max(num / den) < 5 * tol, "worst row %d: %.3e" % (np.argmax(num / den), np.max(num / den))
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse))
    # the kernel feeds the tensor cores bf16 copies of the rotated query and
    # window keys: a relative 2^-8 on the rotated part of each logit
    extra = np.broadcast_to(np.asarray(lse_extra, dtype=np.float64), rl.shape)
    assert np.all(np.abs(lse[fin] - rl[fin]) < 2e-2 + 4e-3 * np.abs(rl[fin]) + extra[fin])


def check_layer_sampled_rows(p, x, outs, rows, f, iqp, b=0, tol=1e-2):
    """Oracle check of batch element b of a whole-layer call on sampled query
    rows, all heads: the stored entries (and index keys), the top-K sets of
    those rows (>= 99% agreement, and at most two swaps in the tie band, none
    outside the strict 1e-6 * |I_K| band beyond two), o and lse, and the
    projected rows y when the call made them.

    x: the layer's inputs (any device); outs: its outputs; iqp: the
    library's own prepared indexer queries [B, S, Hi, Di] (CSA), for the
    stage-wise selection check; f: the rotary inverse frequencies.
    """
    sl = slice(b, b + 1)
    K = p["K"]
    rws = torch.from_numpy(np.asarray(rows)).to(x["q"].device)
    ent = None
    if p["ratio"] > 0:
        ent = O.compress(np64(x["ckv"][sl]), np64(x["cscore"][sl]), np64(x["ape"]), None, f, p["ratio"],
                         p["overlap"], 1e-6, store_bf16=True)
        assert rel_l2(np64(outs["ent"][sl]), ent) < 1e-3
    idx_rows = None
    if K:
        ikey = O.compress(np64(x["ickv"][sl]), np64(x["icscore"][sl]), np64(x["iape"]), None, f, p["ratio"],
                          p["overlap"], 1e-6, hadamard=True, store_bf16=True)
        assert rel_l2(np64(outs["ikey"][sl]), ikey) < 1e-3
        iq_rows = np64(x["iq"][sl][:, rws])
        w_rows = np64(x["w"][sl][:, rws])
        sel = O.indexer_topk(iq_rows, ikey, w_rows, f, p["ratio"], K, store_bf16=True, rows=rows, rows_only=True)
        gi = outs["idx"][b, rws.to(outs["idx"].device)].cpu().numpy()
        agree = total = 0
        for i in range(len(rows)):
            a = set(gi[i][gi[i] >= 0].tolist())
            r = set(sel["idx"][0, i][sel["idx"][0, i] >= 0].tolist())
            assert len(a) == len(r)
            agree += len(a & r)
            total += len(r)
        assert agree >= 0.99 * total, (agree, total)
        idx_rows = sel["idx"]
        # stage-wise: the oracle's scores of the library's own prepared
        # queries and index keys select the same sets outside the tie band
        iqp_rows = np64(iqp[sl][:, rws.to(iqp.device)])
        ikey_g = np64(outs["ikey"][sl])
        sc = O.indexer_scores(iqp_rows, ikey_g, w_rows, p["ratio"], rows=rows, rows_only=True)[0]
        S = p["S"]
        iqp_full = np.zeros((S,) + iqp_rows.shape[2:])
        iqp_full[rows] = iqp_rows[0]
        w_full = np.zeros((S, p["Hi"]))
        w_full[rows] = w_rows[0]
        swaps, wide = check_topk_rows(gi, sc, iqp_full, ikey_g[0], w_full, p["ratio"], K, rows,
                                      O.indexer_scale(p["Hi"], p["Di"]), detail=True)
        print("batch %d sampled rows: in-band swaps %d, swaps outside 1e-6*|I_K| %d" % (b, swaps, wide))
        assert swaps <= 2, swaps
        assert wide <= 2, wide            # only the fp32 error bound would allow these
    q_rows = np64(x["q"][sl][:, rws])
    # the oracle attends with its own entries and its own selection
    ro, rl = O.sparse_mqa(q_rows, np64(x["kv"][sl]), ent, idx_rows, None, f, p["ratio"], p["W"],
                          store_bf16=True, rows=rows, rows_only=True)
    go = np64(outs["o"][sl][:, rws.to(outs["o"].device)])
    gl = np64(outs["lse"][sl][:, rws.to(outs["lse"].device)])
    check_attention_rows(go, gl, ro, rl, tol)
    if "y" in outs:
        ry = O.grouped_wo_a(ro, np64(x["wo_a"]), store_bf16=True)
        gy = np64(outs["y"][sl][:, rws.to(outs["y"].device)])
        assert rel_l2(gy, ry) < tol
        num = np.linalg.norm((gy - ry).reshape(len(rows), -1), axis=1)
        den = np.linalg.norm(ry.reshape(len(rows), -1), axis=1) + 1e-30
        assert np.max(num / den) < 5 * tol
