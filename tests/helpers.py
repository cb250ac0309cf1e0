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
