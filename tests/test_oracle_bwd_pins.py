"""Pins of the oracle's attention backward against things other than itself.

* central differences of the oracle's forward (float64) on tiny layers of the
  three kinds (selected entries + window + sink, all entries, window only);
* torch autograd through scaled_dot_product_attention (float64, CPU) where the
  layer reduces to causal or sliding-window MQA;
* linearity in the queries: the contributions of disjoint row sets add up;
* planted mistakes in the backward's source, each caught by the first pin.
"""
import inspect
import textwrap

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import v4_oracle as O

RNG = np.random.default_rng(4321)


def _layer(kind, S=10, H=2, D=8, R=4, seed=0):
    rng = np.random.default_rng(seed)
    f = O.make_inv_freq(10000.0, R) if R else np.zeros(0, dtype=np.float32)
    x = dict(q=rng.standard_normal((1, S, H, D)), kv=rng.standard_normal((1, S, D)),
             dout=rng.standard_normal((1, S, H, D)), f=f, ent=None, idx=None, sink=None)
    if kind == "csa":
        x.update(ratio=2, window=3, sink=rng.standard_normal(H) * 0.5)
        N = S // 2
        x["ent"] = rng.standard_normal((1, N, D))
        K = 3
        idx = np.full((1, S, K), -1, dtype=np.int32)
        for t in range(S):
            nv = O.n_visible(t, 2)
            take = min(K, nv)
            idx[0, t, rng.permutation(K)[:take]] = rng.permutation(nv)[:take]
        x["idx"] = idx
    elif kind == "hca":
        x.update(ratio=3, window=2, sink=None)
        x["ent"] = rng.standard_normal((1, S // 3, D))
    else:
        x.update(ratio=0, window=-1, sink=rng.standard_normal(H) * 0.5)
    return x


def _loss(x, **over):
    y = dict(x, **over)
    o, _ = O.sparse_mqa(y["q"], y["kv"], y["ent"], y["idx"], y["sink"], y["f"], y["ratio"], y["window"])
    return float((o * y["dout"]).sum())


def _central(x, name, eps=1e-6):
    base = np.array(x[name], dtype=np.float64)
    g = np.zeros_like(base)
    it = np.nditer(base, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        hi, lo = base.copy(), base.copy()
        hi[i] += eps
        lo[i] -= eps
        g[i] = (_loss(x, **{name: hi}) - _loss(x, **{name: lo})) / (2 * eps)
    return g


def _bwd(x):
    return O.sparse_mqa_bwd(x["q"], x["kv"], x["ent"], x["idx"], x["sink"], x["f"], x["ratio"], x["window"],
                            x["dout"])


@pytest.mark.parametrize("kind", ["csa", "hca", "swa"])
def test_bwd_matches_central_differences(kind):
    x = _layer(kind)
    dq, dkv, dent, dsink = _bwd(x)
    np.testing.assert_allclose(dq, _central(x, "q"), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dkv, _central(x, "kv"), rtol=1e-6, atol=1e-7)
    if x["ent"] is not None:
        np.testing.assert_allclose(dent, _central(x, "ent"), rtol=1e-6, atol=1e-7)
    if x["sink"] is not None:
        np.testing.assert_allclose(dsink, _central(x, "sink"), rtol=1e-6, atol=1e-7)
    # every gradient is exercised (no silently zero output)
    assert np.abs(dq).max() > 1e-3 and np.abs(dkv).max() > 1e-3


@pytest.mark.parametrize("window", [-1, 5])
def test_bwd_matches_sdpa_autograd(window):
    # no rotation, no entries, no sink: causal (or sliding-window) MQA with
    # K = V = kv shared by the heads
    S, H, D = 24, 3, 16
    q = RNG.standard_normal((1, S, H, D))
    kv = RNG.standard_normal((1, S, D))
    dout = RNG.standard_normal((1, S, H, D))
    f = np.zeros(0, dtype=np.float32)
    dq, dkv, dent, dsink = O.sparse_mqa_bwd(q, kv, None, None, None, f, 0, window, dout)
    assert dent is None and dsink is None
    qt = torch.tensor(q[0].transpose(1, 0, 2), requires_grad=True)            # [H,S,D]
    kt = torch.tensor(kv[0], requires_grad=True)                              # [S,D]
    i = torch.arange(S)
    mask = i[None, :] <= i[:, None]
    if window > 0:
        mask &= i[None, :] > i[:, None] - window
    k3 = kt[None].expand(H, S, D)
    out = F.scaled_dot_product_attention(qt, k3, k3, attn_mask=mask, scale=D ** -0.5)
    out.backward(torch.from_numpy(dout[0].transpose(1, 0, 2)))
    np.testing.assert_allclose(dq[0], qt.grad.numpy().transpose(1, 0, 2), atol=1e-12)
    np.testing.assert_allclose(dkv[0], kt.grad.numpy(), atol=1e-12)


def test_bwd_rows_add_up():
    x = _layer("csa", S=12)
    full = _bwd(x)
    parts = [O.sparse_mqa_bwd(x["q"], x["kv"], x["ent"], x["idx"], x["sink"], x["f"], x["ratio"], x["window"],
                              x["dout"], rows=r) for r in (np.arange(0, 5), np.arange(5, 12))]
    np.testing.assert_allclose(np.concatenate([p[0] for p in parts], axis=1), full[0], atol=1e-13)
    for k in (1, 2, 3):
        np.testing.assert_allclose(parts[0][k] + parts[1][k], full[k], atol=1e-13)


def test_bwd_empty_key_set_gives_zero():
    # window 0 and no visible entry: the output is 0 whatever q, so dq = 0
    x = _layer("hca", S=4)
    x["window"] = 0
    dq, dkv, dent, _ = _bwd(x)
    assert np.all(dq[0, :2] == 0.0)           # t = 0, 1 see no entry (ratio 3)
    assert np.all(dkv == 0.0)


# ------------------------------------------------------------ planted mistakes
_MUTATIONS = {
    "delta dropped": ("g @ keys.T - delta[:, None]", "g @ keys.T"),
    "dq not de-rotated": ("dq[b, i] = rope_derotate(scale * (ds @ keys), t, inv_freq)",
                          "dq[b, i] = scale * (ds @ keys)"),
    "value path dropped": ("dk = scale * (ds.T @ qr) + p.T @ g", "dk = scale * (ds.T @ qr)"),
    "scale dropped in dk": ("dk = scale * (ds.T @ qr) + p.T @ g", "dk = (ds.T @ qr) + p.T @ g"),
    "window grad not de-rotated": ("rope_derotate(dk[ns:], u, inv_freq)", "dk[ns:]"),
    "sink sign": ("dsink -= ", "dsink += "),
    "dout not rotated": ("g = rope_rotate(dout[b, t], t, inv_freq)", "g = dout[b, t]"),
}


@pytest.mark.parametrize("name", sorted(_MUTATIONS))
def test_central_difference_pin_catches_planted_mistake(monkeypatch, name):
    old, new = _MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(O.sparse_mqa_bwd))
    assert old in src, name
    ns = dict(vars(O))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    monkeypatch.setattr(O, "sparse_mqa_bwd", ns["sparse_mqa_bwd"])
    with pytest.raises(AssertionError):
        test_bwd_matches_central_differences("csa")
