"""Grouped low-rank output projection (tcgen05 GEMM) against the oracle, alone
and as the last step of a layer call."""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from oracle import v4_oracle as O
from tests.helpers import inv_freq_for, np64, oracle_inputs, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,S", [(1, 128), (2, 150), (1, 600)])
def test_grouped_projection_matches_oracle(B, S):
    p = SI.preset("csa_bf16_4k", B=B, S=S, q_mode="direct")
    g = torch.Generator(device="cpu").manual_seed(5)
    o = (torch.randn(B, S, 64, 512, generator=g) * 0.5).to(torch.bfloat16)
    wa = (torch.randn(8, 4096, 1024, generator=g) * 0.02).to(torch.bfloat16)
    y = torch.empty(B, S, 8192, dtype=torch.bfloat16, device="cuda")
    cfg = V.config_from_preset(p)
    V.v4_grouped_o_proj(cfg, o.cuda(), wa.cuda(), y)
    torch.cuda.synchronize()
    ref = O.grouped_wo_a(np64(o), np64(wa), store_bf16=True)
    got = np64(y)
    assert rel_l2(got, ref) < 1e-2
    # every output row, and bf16 rounding of an fp32 sum (K = 4096 terms)
    num = np.linalg.norm((got - ref).reshape(B * S, -1), axis=1)
    den = np.linalg.norm(ref.reshape(B * S, -1), axis=1)
    assert np.max(num / den) < 1e-2


def test_layer_with_projection():
    p = SI.preset("hca_bf16_16k", S=300, q_mode="direct")
    x = SI.make_layer_inputs(p, "cpu", seed=2, wo_a=True)
    f = inv_freq_for(p)
    xd = to_dev(x)
    xd["inv_freq"] = torch.from_numpy(f).cuda()
    cfg = V.config_from_preset(p)
    outs = {"o": torch.empty_like(xd["q"]),
            "y": torch.empty(1, 300, 8192, dtype=torch.bfloat16, device="cuda")}
    V.v4_attn_layer_fwd(cfg, xd, outs, V.alloc_workspace(cfg))
    torch.cuda.synchronize()
    ref = O.attn_layer(dict(ratio=p["ratio"], overlap=p["overlap"], window=p["W"], topk=0, rms_eps=1e-6,
                            store_bf16=True), oracle_inputs(x, f))
    assert rel_l2(np64(outs["o"]), ref["o"]) < 1e-2
    assert rel_l2(np64(outs["y"]), ref["y"]) < 1e-2


def test_unsupported_projection_shape_is_rejected():
    p = SI.preset("csa_bf16_4k", S=64, q_mode="direct")
    cfg = V.config_from_preset(p)
    cfg.o_rank = 1000
    with pytest.raises(V.V4Error) as e:
        V.v4_grouped_o_proj(cfg, torch.empty(1, 64, 64, 512, dtype=torch.bfloat16, device="cuda"),
                            torch.empty(8, 4096, 1000, dtype=torch.bfloat16, device="cuda"),
                            torch.empty(1, 64, 8000, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == 2
