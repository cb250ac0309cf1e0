"""Sparse indexer distillation target on the GPU against the oracle.

The GPU forward gives lse; the target kernel recomputes the selected
entries' logits on the tensor cores, sums the heads' probabilities and the
row pass normalises them, forms the indexer's softmax, the KL loss and its
gradient.  The oracle computes its own float64 attention from the same
inputs.  Cases: selections over several 128-entry tiles with padding slots
in random positions, rows without selections, a sink and a short window,
two batches, 128 and 192 heads (slices summed), top-1024, and ~510 sampled
rows of the S=16384 layer.  Tolerance: 1e-2 relative L2 for the target and
the gradient (bf16 queries and entries, fp32 accumulation), and the loss
within 1e-2 relative plus 1e-4 absolute.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from oracle import v4_oracle as O
from tests.helpers import inv_freq_for, np64, rel_l2

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_compressed_attention_gb300 import build
    build.build()


def _gpu_target(p, sink, seed=0, idx_seed=7):
    x = SI.make_layer_inputs(p, "cuda", seed=seed, sink=sink)
    ent = SI.make_entries(p, "cuda", seed=seed + 3)
    B, S, H, K, r = p["B"], p["S"], p["H"], p["K"], p["ratio"]
    idx = SI.random_topk_indices(B, S, r, K, "cpu", seed=idx_seed)
    g = torch.Generator(device="cpu").manual_seed(seed + 11)
    isc = torch.randn(B, S, K, generator=g) * 2.0
    isc[idx < 0] = float("-inf")
    f = inv_freq_for(p)
    fd = torch.from_numpy(f).cuda()
    cfg = V.config_from_preset(p, path=V.V4_PATH_TC)
    ws = V.alloc_workspace(cfg)
    o = torch.empty_like(x["q"])
    lse = torch.empty(B, S, H, device="cuda")
    V.v4_reset_device_status()
    V.v4_sparse_mqa_fwd(cfg, x["q"], x["kv"], ent, idx.cuda(), x["sink"], fd, o, lse, ws)
    target = torch.full((B, S, K), float("nan"), device="cuda")
    loss = torch.full((B, S), float("nan"), device="cuda")
    dscore = torch.full((B, S, K), float("nan"), device="cuda")
    V.v4_indexer_kl_target(cfg, x["q"], ent, idx.cuda(), lse, isc.cuda(), fd, target, loss, dscore, ws)
    torch.cuda.synchronize()
    assert V.v4_get_device_status() == 0
    host = dict(q=np64(x["q"]), kv=np64(x["kv"]), ent=np64(ent), idx=idx.numpy(), sink=np64(x["sink"]),
                isc=isc.numpy().astype(np.float64), f=f)
    return host, dict(target=np64(target), loss=np64(loss), dscore=np64(dscore))


def _oracle(p, h, rows=None):
    return O.indexer_kl_target(h["q"], h["kv"], h["ent"], h["idx"], h["sink"], h["f"], p["ratio"], p["W"],
                               iscore=h["isc"], rows=rows)


def _check(g, ref, idx):
    assert np.all(np.isfinite(g["target"])) and np.all(np.isfinite(g["dscore"])) and np.all(np.isfinite(g["loss"]))
    assert np.all(g["target"][idx < 0] == 0) and np.all(g["dscore"][idx < 0] == 0)
    assert rel_l2(g["target"], ref["target"]) < TOL, rel_l2(g["target"], ref["target"])
    assert rel_l2(g["dscore"], ref["dscore"]) < TOL, rel_l2(g["dscore"], ref["dscore"])
    assert np.all(np.abs(g["loss"] - ref["loss"]) <= TOL * np.abs(ref["loss"]) + 1e-4)
    valid_rows = (idx >= 0).any(axis=-1)
    np.testing.assert_allclose(g["target"].sum(axis=-1)[valid_rows], 1.0, rtol=1e-4)


CASES = [
    ("k64_s700", dict(S=700, K=64), False),
    ("k512_s2100_sink", dict(S=2100), True),
    ("k32_b2_w37_sink", dict(S=300, B=2, K=32, W=37), True),
    ("h128_k1024", dict(S=1300, H=128, K=1024), False),
    ("h192_b2", dict(S=200, B=2, H=192, K=40), True),
]


@pytest.mark.parametrize("name,over,sink", CASES, ids=[c[0] for c in CASES])
def test_kl_target_matches_oracle(name, over, sink):
    p = SI.preset("csa_bf16_4k", **over)
    h, g = _gpu_target(p, sink)
    _check(g, _oracle(p, h), h["idx"])


def test_full_size_sampled_rows():
    p = SI.preset("csa_bf16_16k")
    h, g = _gpu_target(p, sink=False, seed=5)
    S = p["S"]
    rows = np.unique(np.concatenate([np.linspace(0, S - 1, 504).round().astype(int), [1, 3, 4, 127, 4096, S - 2]]))
    ref = _oracle(p, h, rows=rows)
    sub = {k: g[k][:, rows] for k in g}
    _check(sub, ref, h["idx"][:, rows])


def test_rejects_unsupported_shapes():
    p = SI.preset("tiny_csa_f32")
    cfg = V.config_from_preset(p)
    B, S, K = p["B"], p["S"], p["K"]
    with pytest.raises(V.V4Error) as e:
        V.v4_indexer_kl_target(cfg, torch.empty(B, S, p["H"], p["D"], device="cuda"),
                               torch.empty(B, S // p["ratio"], p["D"], device="cuda"),
                               torch.zeros(B, S, K, dtype=torch.int32, device="cuda"),
                               torch.zeros(B, S, p["H"], device="cuda"), None, None,
                               torch.empty(B, S, K, device="cuda"), None, None, V.alloc_workspace(cfg))
    assert e.value.status == 2
