"""Tensor-core attention (tcgen05 / TMA) against the oracle.

Forced tensor-core path at the Flash shapes (64 heads, 512-d latent, 64 rotated
dims, bf16): CSA selections, HCA dense entries, window-only, ragged lengths,
batches, sink, top-512 over several entry tiles, inputs whose large norms push
the softmax bound far above the logits (those queries go through the
running-max fix-up), and the full S=16384 layers of the benchmark checked on
sampled rows.  Tolerance: 1e-2 relative L2 (bf16 storage, fp32 accumulation).
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from oracle import v4_oracle as O
from tests.helpers import check_attention_rows, check_layer_sampled_rows, inv_freq_for, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_compressed_attention_gb300 import build
    build.build()
    V.lib()


def _run(p, mode, sink, path, seed=0, q_scale=1.0, idx_seed=7, kv_scale=1.0):
    x = SI.make_layer_inputs(p, "cpu", seed=seed, sink=sink)
    if q_scale != 1.0:
        x["q"] = (x["q"].float() * q_scale).to(x["q"].dtype)
    if kv_scale != 1.0:
        x["kv"] = (x["kv"].float() * kv_scale).to(x["kv"].dtype)
    f = inv_freq_for(p)
    xd = to_dev(x)
    fd = torch.from_numpy(f).cuda()
    B, S, H, r = p["B"], p["S"], p["H"], p["ratio"]
    ent = ent_d = idx = idx_d = None
    if r > 0:
        ent = O.compress(np64(x["ckv"]), np64(x["cscore"]), np64(x["ape"]), None, f, r, p["overlap"],
                         1e-6, store_bf16=True)
        ent_d = torch.from_numpy(ent).to(torch.bfloat16).cuda()
    K = p["K"] if mode == "csa" else 0
    if mode == "csa":
        idx_d = SI.random_topk_indices(B, S, r, K, "cpu", seed=idx_seed)
        idx = idx_d.numpy()
        idx_d = idx_d.cuda()
    cfg = V.config_from_preset(p, K=K, path=path)
    o = torch.empty_like(xd["q"])
    lse = torch.empty(B, S, H, dtype=torch.float32, device="cuda")
    ws = V.alloc_workspace(cfg)
    V.v4_reset_device_status()
    V.v4_sparse_mqa_fwd(cfg, xd["q"], xd["kv"], ent_d, idx_d, xd["sink"], fd, o, lse, ws)
    assert V.v4_get_device_status() == 0
    ro, rl = O.sparse_mqa(np64(x["q"]), np64(x["kv"]), ent, idx, np64(x["sink"]), f, r, p["W"],
                          store_bf16=True)
    return np64(o), np64(lse), ro, rl


def _check(o, lse, ro, rl, tol=TOL):
    check_attention_rows(o, lse, ro, rl, tol)


CASES = [
    # name, preset, overrides, mode, sink
    ("csa_k64_s700", "csa_bf16_4k", dict(S=700, K=64), "csa", False),
    ("csa_k512_s2100", "csa_bf16_4k", dict(S=2100), "csa", False),
    ("csa_k32_b2_sink", "csa_bf16_4k", dict(S=300, B=2, K=32), "csa", True),
    ("csa_s1", "csa_bf16_4k", dict(S=1, K=16), "csa", False),
    ("hca_s1000_sink", "hca_bf16_16k", dict(S=1000), "hca", True),
    ("hca_two_tiles", "hca_bf16_16k", dict(S=260, ratio=2), "hca", False),
    ("hca_b2_ragged", "hca_bf16_16k", dict(S=777, B=2, ratio=16), "hca", False),
    ("swa_s300", "swa_bf16_16k", dict(S=300), "swa", False),
    ("swa_w7_b2", "swa_bf16_16k", dict(S=100, B=2, W=7), "swa", True),
    # V4-Pro-like shapes: 128 heads (two 64-head slices per query), top-1024
    ("pro_csa_h128_k1024_sink", "csa_bf16_4k", dict(S=4500, H=128, K=1024), "csa", True),
    ("pro_hca_h128", "hca_bf16_16k", dict(S=700, H=128), "hca", False),
    ("csa_h192_b2", "csa_bf16_4k", dict(S=400, B=2, H=192, K=96), "csa", False),
]


@pytest.mark.parametrize("name,base,over,mode,sink", CASES, ids=[c[0] for c in CASES])
def test_tc_attention_matches_oracle(name, base, over, mode, sink):
    p = SI.preset(base, q_mode="direct", **over)
    o, lse, ro, rl = _run(p, mode, sink, V.V4_PATH_TC)
    _check(o, lse, ro, rl)


def test_tc_and_simt_agree():
    p = SI.preset("csa_bf16_4k", q_mode="direct", S=900, K=128)
    o1, l1, ro, rl = _run(p, "csa", True, V.V4_PATH_TC)
    o2, l2, _, _ = _run(p, "csa", True, V.V4_PATH_SIMT)
    assert rel_l2(o1, o2) < TOL
    _check(o2, l2, ro, rl)


def test_large_norms_take_the_fixup_path():
    # q scaled by 16: logits spread over hundreds, so a window key can rise
    # far above the shift taken from the entry tile; queries whose
    # denominator overflows the check are recomputed with a running max.
    p = SI.preset("hca_bf16_16k", q_mode="direct", S=400, ratio=16)
    o, lse, ro, rl = _run(p, "hca", False, V.V4_PATH_TC, q_scale=16.0)
    _check(o, lse, ro, rl)


def test_keys_far_above_the_first_tile_take_the_fixup_path():
    # Window keys scaled by 64 (entries, from their own RMSNormed pooling,
    # are not): for every query with entries the window logits exceed the
    # first (entry) tile's maximum by far more than exp's range, so the
    # shifted exponentials overflow; only the running-max fix-up of those
    # queries gives finite, correct outputs.
    p = SI.preset("hca_bf16_16k", q_mode="direct", S=400, ratio=16)
    o, lse, ro, rl = _run(p, "hca", False, V.V4_PATH_TC, kv_scale=64.0)
    assert np.all(np.isfinite(o))
    # Both kernels read bf16 copies of the rotated query and window keys: a
    # logit may move by up to scale * 2^-8 * |q_rot| * |k_rot|, which the
    # 64-fold keys make larger than the unit-scale allowance of lse.
    x = SI.make_layer_inputs(p, "cpu", seed=0)
    R = p["R"]
    q_rot = np.linalg.norm(np64(x["q"])[..., -R:], axis=-1)                 # [B, S, H]
    k_rot = np.linalg.norm(np64(x["kv"])[..., -R:], axis=-1).max() * 64.0
    extra = 2.0 ** -8 * q_rot * k_rot / np.sqrt(p["D"])
    check_attention_rows(o, lse, ro, rl, TOL, lse_extra=extra)


def test_forced_tc_path_rejects_other_shapes():
    p = SI.preset("tiny_csa_f32", ratio=0, overlap=0, K=0)
    cfg = V.config_from_preset(p, path=V.V4_PATH_TC)
    x = SI.make_layer_inputs(p, "cuda")
    with pytest.raises(V.V4Error) as e:
        V.v4_sparse_mqa_fwd(cfg, x["q"], x["kv"], None, None, None,
                            torch.from_numpy(inv_freq_for(p)).cuda(), torch.empty_like(x["q"]), None,
                            V.alloc_workspace(cfg))
    assert e.value.status == 2


@pytest.mark.parametrize("name", ["csa_bf16_16k", "hca_bf16_16k"])
def test_full_size_layer_sampled_rows(name):
    """The bench's layers (B=1, S=16384, rank-1024 queries) through
    v4_attn_layer_fwd, checked on ~510 sampled query rows, all heads (and,
    for CSA, the top-512 sets of those rows), with the full compressor."""
    p = SI.preset(name)
    x = SI.make_layer_inputs(p, "cuda", seed=11)
    f = inv_freq_for(p)
    xd = dict(x, inv_freq=torch.from_numpy(f).cuda())
    cfg = V.config_from_preset(p)
    B, S, H, K = p["B"], p["S"], p["H"], p["K"]
    outs = {"o": torch.empty_like(x["q"]), "lse": torch.empty(B, S, H, device="cuda")}
    if K:
        outs["idx"] = torch.empty(B, S, K, dtype=torch.int32, device="cuda")
        outs["ikey"] = torch.empty(B, S // p["ratio"], p["Di"], dtype=torch.bfloat16, device="cuda")
    outs["ent"] = torch.empty(B, S // p["ratio"], p["D"], dtype=torch.bfloat16, device="cuda")
    ws = V.alloc_workspace(cfg)
    V.v4_reset_device_status()
    V.v4_attn_layer_fwd(cfg, xd, outs, ws)
    torch.cuda.synchronize()
    assert V.v4_get_device_status() == 0
    rows = np.unique(np.concatenate([np.linspace(0, S - 1, 504).round().astype(int),
                                     [0, 1, 127, 128, 511, 512, 2047, S - 1]]))
    iqp = V.v4_indexer_prep(cfg, x["iq"], xd["inv_freq"], torch.empty_like(x["iq"])) if K else None
    check_layer_sampled_rows(p, x, outs, rows, f, iqp)
