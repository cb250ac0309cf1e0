"""Query-row slices of one sequence through the C ABI (one GPU).

A call with q_begin = a and seqlen = b computes query positions a..b-1 from
the sequence's first b tokens (causality: no later token is read).  The
slices of a zig-zag split must reproduce the whole-sequence call bit for bit:
every query row is computed by the same kernels with the same arithmetic,
only the rows a call owns change.  This is what lets one sequence spread over
several GPUs without any exchange on the data path.
"""
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from sparse_compressed_attention_gb300 import rows as R
from tests.helpers import inv_freq_for

pytestmark = pytest.mark.gpu

ROW_IN = ("q", "iq", "w")                        # one row per query position
SEQ_IN = ("kv", "ckv", "cscore", "ickv", "icscore")


def _outputs(p, rows, wo_a):
    B, H, D, K = p["B"], p["H"], p["D"], p["K"]
    dt = SI.torch_dtype(p)
    o = {"o": torch.empty(B, rows, H, D, dtype=dt, device="cuda"),
         "lse": torch.empty(B, rows, H, device="cuda")}
    if K > 0:
        o["idx"] = torch.empty(B, rows, K, dtype=torch.int32, device="cuda")
        o["iscore"] = torch.empty(B, rows, K, device="cuda")
    if wo_a is not None:
        o["y"] = torch.empty(B, rows, wo_a.shape[0] * wo_a.shape[2], dtype=dt, device="cuda")
    return o


def _run(p, x, a, b, **cfg_over):
    cfg = V.config_from_preset(p, S=b, q_begin=a, **cfg_over)
    xi = {}
    for k, v in x.items():
        if k in ROW_IN and v is not None:
            xi[k] = v[:, a:b].clone()            # own allocation: 16-byte aligned
        elif k in SEQ_IN and v is not None:
            xi[k] = v[:, :b].contiguous()
        else:
            xi[k] = v
    out = _outputs(p, b - a, x.get("wo_a"))
    V.v4_attn_layer_fwd(cfg, xi, out, V.alloc_workspace(cfg))
    return out


CASES = [
    ("csa_bf16", "csa_bf16_4k", dict(S=4096, q_mode="direct"), 2, {}),
    ("csa_bf16_b2", "csa_bf16_4k", dict(B=2, S=1500, q_mode="direct"), 3, {}),
    ("csa_e4m3", "csa_bf16_4k", dict(S=2048, q_mode="direct"), 2, dict(indexer_fp8=1)),
    ("hca_bf16_wo_a", "hca_bf16_16k", dict(S=3000, q_mode="direct"), 4, {}),
    ("swa_bf16", "swa_bf16_16k", dict(S=1000, q_mode="direct"), 2, {}),
    ("tiny_f32", "tiny_csa_f32", dict(), 2, {}),
]


@pytest.mark.parametrize("name,base,over,world,cfg_over", CASES, ids=[c[0] for c in CASES])
def test_row_slices_equal_the_whole_sequence(name, base, over, world, cfg_over):
    from sparse_compressed_attention_gb300 import build
    build.build()
    p = SI.preset(base, **over)
    x = SI.make_layer_inputs(p, "cuda", seed=21, sink=True, wo_a=name.endswith("wo_a"))
    x["inv_freq"] = torch.from_numpy(inv_freq_for(p)).cuda()
    S = p["S"]
    whole = _run(p, x, 0, S, **cfg_over)
    cost = R.layer_cost(p["ratio"], p["K"], p["W"], heads=p["H"], dim=p["D"], idx_heads=p["Hi"], idx_dim=p["Di"])
    covered = torch.zeros(S, dtype=torch.int32)
    for rank in range(world):
        for a, b in R.zigzag_chunks(S, world, rank, cost):
            part = _run(p, x, a, b, **cfg_over)
            covered[a:b] += 1
            for k, v in part.items():
                ref = whole[k][:, a:b]
                assert torch.equal(v, ref), (name, rank, a, b, k)
    assert torch.equal(covered, torch.ones(S, dtype=torch.int32))
    assert V.v4_get_device_status() == 0
