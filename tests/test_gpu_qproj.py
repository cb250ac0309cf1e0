"""Query projections of the rank-1024 latent (tcgen05 GEMM, per-head RMSNorm
epilogue) against the oracle: ragged token counts across 128-row tiles,
with and without a norm weight, the indexer queries from the same latent,
another rank; then the layer fed the projected queries agrees with the
oracle fed the oracle's.  Tolerance: every element within 2 bf16 ulps of
the oracle's rounded value plus the fp32 error of a K-term sum, and 1e-2
relative L2."""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from oracle import v4_oracle as O
from tests.helpers import assert_within_bf16_ulp, np64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_compressed_attention_gb300 import build
    build.build()


def _draw(B, S, rank, n_out, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    qlat = torch.randn(B, S, rank, generator=g).to(torch.bfloat16)
    w = (torch.randn(rank, n_out, generator=g) * 0.02).to(torch.bfloat16)
    return qlat, w


def _check(got, ref, rank):
    assert rel_l2(got, ref) < 1e-2
    # an fp32 sum of `rank` products, then (with the norm) a scale: allow the
    # sum's forward error relative to the row magnitude on top of 2 ulps
    assert_within_bf16_ulp(got, ref, ulps=2, row_terms=rank + 8)


@pytest.mark.parametrize("B,S,norm_w", [(1, 128, False), (2, 300, True), (1, 1, False)])
def test_q_projection_matches_oracle(B, S, norm_w):
    p = SI.preset("csa_bf16_4k", B=B, S=S, q_mode="direct")
    H, D, rank = p["H"], p["D"], 1024
    qlat, wq = _draw(B, S, rank, H * D, seed=S)
    gw = torch.linspace(0.5, 1.5, D) if norm_w else None
    cfg = V.config_from_preset(p)
    q = torch.empty(B, S, H, D, dtype=torch.bfloat16, device="cuda")
    V.v4_q_proj(cfg, qlat.cuda(), wq.cuda(), q, q_norm=1, q_norm_w=gw.cuda() if norm_w else None)
    torch.cuda.synchronize()
    assert V.v4_get_device_status() == 0
    ref = O.q_projection(np64(qlat), np64(wq), H, D, norm=True, eps=cfg.rms_eps,
                         norm_w=np64(gw) if norm_w else None, store_bf16=True)
    _check(np64(q), ref, rank)
    np.testing.assert_allclose(np.sqrt(np.mean(np64(q) ** 2, axis=-1)) if not norm_w else 1.0, 1.0, rtol=1e-2)


def test_indexer_queries_from_the_same_latent():
    p = SI.preset("csa_bf16_4k", B=1, S=257, q_mode="direct")
    H, D, Hi, Di, rank = p["H"], p["D"], p["Hi"], p["Di"], 1024
    qlat, wq = _draw(1, 257, rank, H * D, seed=3)
    _, wiq = _draw(1, 1, rank, Hi * Di, seed=4)
    cfg = V.config_from_preset(p)
    q = torch.empty(1, 257, H, D, dtype=torch.bfloat16, device="cuda")
    iq = torch.empty(1, 257, Hi, Di, dtype=torch.bfloat16, device="cuda")
    V.v4_q_proj(cfg, qlat.cuda(), wq.cuda(), q, q_norm=0, wiq=wiq.cuda(), iq=iq)
    torch.cuda.synchronize()
    _check(np64(q), O.q_projection(np64(qlat), np64(wq), H, D, norm=False, store_bf16=True), rank)
    _check(np64(iq), O.indexer_q_projection(np64(qlat), np64(wiq), Hi, Di, store_bf16=True), rank)


def test_other_rank_and_width():
    p = SI.preset("hca_bf16_16k", B=1, S=200, H=128, q_mode="direct")
    H, D, rank = p["H"], p["D"], 320
    qlat, wq = _draw(1, 200, rank, H * D, seed=9)
    cfg = V.config_from_preset(p)
    q = torch.empty(1, 200, H, D, dtype=torch.bfloat16, device="cuda")
    V.v4_q_proj(cfg, qlat.cuda(), wq.cuda(), q, q_norm=1)
    torch.cuda.synchronize()
    ref = O.q_projection(np64(qlat), np64(wq), H, D, norm=True, eps=cfg.rms_eps, store_bf16=True)
    _check(np64(q), ref, rank)


def test_layer_on_projected_queries():
    """The prologue feeding the layer: the GPU's projected q and iq through
    v4_attn_layer_fwd against the oracle's projections through the oracle's
    layer."""
    p = SI.preset("csa_bf16_4k", S=512, q_mode="direct")
    x = SI.make_layer_inputs(p, "cpu", seed=1)
    H, D, Hi, Di, rank = p["H"], p["D"], p["Hi"], p["Di"], 1024
    qlat, wq = _draw(1, 512, rank, H * D, seed=7)
    _, wiq = _draw(1, 1, rank, Hi * Di, seed=8)
    cfg = V.config_from_preset(p)
    q = torch.empty(1, 512, H, D, dtype=torch.bfloat16, device="cuda")
    iq = torch.empty(1, 512, Hi, Di, dtype=torch.bfloat16, device="cuda")
    V.v4_q_proj(cfg, qlat.cuda(), wq.cuda(), q, q_norm=1, wiq=wiq.cuda(), iq=iq)
    from tests.helpers import inv_freq_for, oracle_inputs, to_dev
    f = inv_freq_for(p)
    xd = dict(to_dev(x), q=q, iq=iq, inv_freq=torch.from_numpy(f).cuda())
    outs = {"o": torch.empty_like(q), "idx": torch.empty(1, 512, p["K"], dtype=torch.int32, device="cuda")}
    V.v4_attn_layer_fwd(cfg, xd, outs, V.alloc_workspace(cfg))
    torch.cuda.synchronize()
    xo = oracle_inputs(x, f)
    xo["q"] = O.q_projection(np64(qlat), np64(wq), H, D, norm=True, eps=cfg.rms_eps, store_bf16=True)
    xo["iq"] = O.indexer_q_projection(np64(qlat), np64(wiq), Hi, Di, store_bf16=True)
    ref = O.attn_layer(dict(ratio=p["ratio"], overlap=p["overlap"], window=p["W"], topk=p["K"], rms_eps=1e-6,
                            store_bf16=True), xo)
    assert rel_l2(np64(outs["o"]), ref["o"]) < 1e-2
