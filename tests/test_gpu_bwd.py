"""Tensor-core attention backward against the oracle's exact gradient.

The GPU backward consumes the GPU forward's o and lse; the oracle computes the
gradient of its own float64 forward from the same seeded inputs (q, kv,
entries, selections, sink, output gradient).  Cases: CSA selections over
several 32-key tiles, HCA dense entries, window-only layers, short windows,
the first query alone, batches, sinks, 128 and 192 heads, top-1024, and the
full S=16384 CSA / HCA layers checked on outputs the oracle can form from a
few hundred queries (dq of sampled queries, dkv of sampled positions, the
gradients of the last entries).  Tolerance: 1e-2 relative L2 (bf16 storage
of q, kv, entries, o, dO, dq and of the tensor-core operands dS and P, fp32
accumulation).
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from oracle import v4_oracle as O
from tests.helpers import inv_freq_for, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_compressed_attention_gb300 import build
    build.build()
    V.lib()


def _gpu_bwd(p, mode, sink, seed=0, idx_seed=7):
    """Forward then backward on the GPU; returns host inputs and GPU results."""
    x = SI.make_layer_inputs(p, "cuda", seed=seed, sink=sink)
    ent = SI.make_entries(p, "cuda", seed=seed + 3) if p["ratio"] > 0 else None
    dout = SI.make_output_grad(p, "cuda", seed=seed + 2)
    f = inv_freq_for(p)
    B, S, H, D, r = p["B"], p["S"], p["H"], p["D"], p["ratio"]
    K = p["K"] if mode == "csa" else 0
    idx = SI.random_topk_indices(B, S, r, K, "cpu", seed=idx_seed) if mode == "csa" else None
    xd = to_dev(dict(q=x["q"], kv=x["kv"], sink=x["sink"], ent=ent, idx=idx, dout=dout))
    fd = torch.from_numpy(f).cuda()
    cfg = V.config_from_preset(p, K=K, path=V.V4_PATH_TC)
    o = torch.empty_like(xd["q"])
    lse = torch.empty(B, S, H, dtype=torch.float32, device="cuda")
    ws = V.alloc_workspace(cfg)
    V.v4_reset_device_status()
    V.v4_sparse_mqa_fwd(cfg, xd["q"], xd["kv"], xd["ent"], xd["idx"], xd["sink"], fd, o, lse, ws)
    dq = torch.empty_like(xd["q"])
    dkv = torch.full((B, S, D), float("nan"), dtype=torch.float32, device="cuda")
    N = ent.shape[1] if ent is not None else 0
    dent = torch.full((B, N, D), float("nan"), dtype=torch.float32, device="cuda") if N > 0 else None
    dsink = torch.full((H,), float("nan"), dtype=torch.float32, device="cuda") if sink else None
    bws = V.alloc_bwd_workspace(cfg)
    V.v4_sparse_mqa_bwd(cfg, xd["q"], xd["kv"], xd["ent"] if N > 0 else None, xd["idx"], xd["sink"], fd, o, lse,
                        xd["dout"], dq, dkv, dent, dsink, bws)
    torch.cuda.synchronize()
    assert V.v4_get_device_status() == 0
    host = dict(q=np64(x["q"]), kv=np64(x["kv"]), ent=np64(ent) if N > 0 else None,
                idx=None if idx is None else idx.numpy(), sink=np64(x["sink"]), dout=np64(dout), f=f)
    gpu = dict(dq=np64(dq), dkv=np64(dkv), dent=np64(dent) if dent is not None else None,
               dsink=np64(dsink) if dsink is not None else None, o=np64(o))
    del xd, o, dq, dkv, dent, dsink, ws, bws
    return host, gpu


def _oracle(p, h, rows=None):
    return O.sparse_mqa_bwd(h["q"], h["kv"], h["ent"], h["idx"], h["sink"], h["f"], p["ratio"], p["W"],
                            h["dout"], rows=rows)


def _rows_check(a, b, tol, floor=None):
    """Relative L2 over everything, and per leading row within 5 * tol of the
    row's norm plus ``floor`` (per row, absolute)."""
    assert np.all(np.isfinite(a))
    a2 = a.reshape(-1, a.shape[-1])
    b2 = b.reshape(-1, b.shape[-1])
    num = np.linalg.norm(a2 - b2, axis=1)
    den = np.linalg.norm(b2, axis=1)
    fl = np.zeros_like(den) if floor is None else np.broadcast_to(np.asarray(floor, dtype=np.float64).ravel(),
                                                                   den.shape)
    # (a one-key softmax has a dq of zero: the oracle's is rounding noise)
    if np.linalg.norm(b) > 1e-6 * np.linalg.norm(fl):
        assert rel_l2(a, b) < tol, rel_l2(a, b)
    # rows the oracle makes (near) zero are judged against the median row
    fl = np.maximum(fl, 1e-3 * np.median(den) + 1e-30)
    excess = num - 5 * tol * den - fl
    if np.any(excess > 0):
        k = int(np.argmax(excess))
        raise AssertionError("%d of %d rows beyond tolerance; worst row %d: err %.3e, norm %.3e, floor %.3e, "
                             "median norm %.3e" % (int(np.sum(excess > 0)), len(den), k, num[k], den[k], fl[k],
                                                   np.median(den)))


def _delta_floor(o, dout, scale):
    """Per (query, head) bound of the dq error that the bf16 output o brings
    in through delta = dO . o: delta is off by at most 2^-8 sum |dO o| (o
    rounded to bf16, fp32 sums), which shifts dq by -scale * err * o' exactly
    (o' = o before de-rotation, same norm); twice that as the allowance."""
    err = 2.0 ** -8 * np.abs(dout * o).sum(axis=-1)
    return 2.0 * scale * err * np.linalg.norm(o, axis=-1)


CASES = [
    # name, preset, overrides, mode, sink
    ("csa_k64_s700", "csa_bf16_4k", dict(S=700, K=64), "csa", False),
    ("csa_k512_s2100_sink", "csa_bf16_4k", dict(S=2100), "csa", True),
    ("csa_k32_b2_sink", "csa_bf16_4k", dict(S=300, B=2, K=32), "csa", True),
    ("csa_s1", "csa_bf16_4k", dict(S=1, K=16), "csa", False),
    ("csa_w37", "csa_bf16_4k", dict(S=400, K=48, W=37), "csa", True),
    ("hca_s1000_sink", "hca_bf16_16k", dict(S=1000), "hca", True),
    ("hca_ratio2_many_tiles", "hca_bf16_16k", dict(S=260, ratio=2), "hca", False),
    ("swa_s500", "swa_bf16_16k", dict(S=500), "swa", True),
    ("swa_w1", "swa_bf16_16k", dict(S=90, W=1), "swa", False),
    ("pro_csa_h128_k1024_sink", "csa_bf16_4k", dict(S=1300, H=128, K=1024), "csa", True),
    ("csa_h192_b2", "csa_bf16_4k", dict(S=200, B=2, H=192, K=40), "csa", True),
]


@pytest.mark.parametrize("name,preset,over,mode,sink", CASES, ids=[c[0] for c in CASES])
def test_bwd_matches_oracle(name, preset, over, mode, sink):
    p = SI.preset(preset, **over)
    h, g = _gpu_bwd(p, mode, sink)
    dq, dkv, dent, dsink = _oracle(p, h)
    _rows_check(g["dq"], dq, TOL, _delta_floor(g["o"], h["dout"], p["D"] ** -0.5))
    _rows_check(g["dkv"], dkv, TOL)
    if dent is not None and dent.size:
        assert g["dent"] is not None
        _rows_check(g["dent"], dent, TOL)
    if sink:
        assert rel_l2(g["dsink"], dsink) < TOL, rel_l2(g["dsink"], dsink)


@pytest.mark.parametrize("preset,mode", [("csa_bf16_16k", "csa"), ("hca_bf16_16k", "hca")])
def test_bwd_full_size_sampled(preset, mode):
    p = SI.preset(preset)
    S, W, r = p["S"], p["W"], p["ratio"]
    h, g = _gpu_bwd(p, mode, sink=False)
    N = S // r
    q_rows = [0, 1, 127, 5000, S // 2 + 3, S - 1]
    u_pos = [0, 9000, S - 200]                       # window positions: rows u .. u + W - 1
    last_e = [N - 1, N - 2]                          # entries read by the last queries only
    e_lo = r * (N - 2) + r - 1                      # first query that sees entry N - 2
    rows = sorted(set(q_rows) | {t for u in u_pos for t in range(u, min(S, u + W))} | set(range(e_lo, S)))
    dq, dkv, dent, _ = _oracle(p, h, rows=np.asarray(rows))
    pos = {t: i for i, t in enumerate(rows)}
    sel = [pos[t] for t in q_rows]
    _rows_check(g["dq"][:, q_rows], dq[:, sel], TOL,
                _delta_floor(g["o"][:, q_rows], h["dout"][:, q_rows], p["D"] ** -0.5))
    _rows_check(g["dkv"][:, u_pos], dkv[:, u_pos], TOL)
    _rows_check(g["dent"][:, last_e], dent[:, last_e], TOL)
    assert np.all(np.isfinite(g["dq"])) and np.all(np.isfinite(g["dkv"])) and np.all(np.isfinite(g["dent"]))


def test_bwd_graph_replay_is_stable():
    # the call is capture-safe; two replays give the same dq (dkv / dent are
    # fp32 reductions in scheduling order, compared with a tolerance)
    p = SI.preset("csa_bf16_4k", S=512, K=64)
    x = SI.make_layer_inputs(p, "cuda", seed=1, sink=True)
    ent = SI.make_entries(p, "cuda", seed=4)
    idx = SI.random_topk_indices(1, 512, 4, 64, "cuda", seed=9)
    dout = SI.make_output_grad(p, "cuda", seed=5)
    fd = torch.from_numpy(inv_freq_for(p)).cuda()
    cfg = V.config_from_preset(p, path=V.V4_PATH_TC)
    o = torch.empty_like(x["q"])
    lse = torch.empty(1, 512, 64, dtype=torch.float32, device="cuda")
    V.v4_sparse_mqa_fwd(cfg, x["q"], x["kv"], ent, idx, x["sink"], fd, o, lse, V.alloc_workspace(cfg))
    dq = torch.empty_like(x["q"])
    dkv = torch.empty(1, 512, 512, device="cuda")
    dent = torch.empty(1, 128, 512, device="cuda")
    dsink = torch.empty(64, device="cuda")
    bws = V.alloc_bwd_workspace(cfg)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        V.v4_sparse_mqa_bwd(cfg, x["q"], x["kv"], ent, idx, x["sink"], fd, o, lse, dout, dq, dkv, dent, dsink, bws)
    st.synchronize()
    ref = [t.clone() for t in (dq, dkv, dent, dsink)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        V.v4_sparse_mqa_bwd(cfg, x["q"], x["kv"], ent, idx, x["sink"], fd, o, lse, dout, dq, dkv, dent, dsink, bws,
                            stream=st)
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(dq, ref[0])
        for a, b in zip((dkv, dent, dsink), ref[1:]):
            assert rel_l2(np64(a), np64(b)) < 1e-5
    assert V.v4_get_device_status() == 0


def test_bwd_rejects_unsupported_shapes():
    # 32 heads: no tensor-core backward for that shape
    p = SI.preset("csa_bf16_4k", S=64, K=16, H=32)
    cfg = V.config_from_preset(p)
    zb = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    zf = torch.zeros(16, device="cuda")
    zi = torch.zeros(16, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(V.V4Error) as e:
        V.v4_sparse_mqa_bwd(cfg, zb, zb, zb, zi, None, zf, zb, zf, zb, zb, zf, zf, None, ws)
    assert e.value.status == 2
