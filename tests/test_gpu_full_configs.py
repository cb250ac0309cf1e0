"""The two largest benchmark configurations through v4_attn_layer_fwd, in the
launch configuration the benchmark times, checked against the oracle on
sampled query rows (all heads): the long-context CSA layer (B=1, S=65536,
top-512 of up to 16384 entries) and the layers of the 43-layer stack (B=2,
S=16384, each followed by the grouped 8 x 1024 output projection), in both
batch elements.  Entries, index keys, the top-512 sets (agreement and
strict-band swap counts), o, lse and the projected rows; tolerance 1e-2
relative L2 (bf16 storage, fp32 accumulation)."""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from tests.helpers import check_layer_sampled_rows, inv_freq_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_compressed_attention_gb300 import build
    build.build()
    V.lib()


def _layer(p, seed, wo_a=False):
    x = SI.make_layer_inputs(p, "cuda", seed=seed, wo_a=wo_a)
    f = inv_freq_for(p)
    xd = dict(x, inv_freq=torch.from_numpy(f).cuda())
    cfg = V.config_from_preset(p)
    B, S, H, K = p["B"], p["S"], p["H"], p["K"]
    outs = {"o": torch.empty_like(x["q"]), "lse": torch.empty(B, S, H, device="cuda")}
    if p["ratio"] > 0:
        outs["ent"] = torch.empty(B, S // p["ratio"], p["D"], dtype=torch.bfloat16, device="cuda")
    if K:
        outs["idx"] = torch.empty(B, S, K, dtype=torch.int32, device="cuda")
        outs["ikey"] = torch.empty(B, S // p["ratio"], p["Di"], dtype=torch.bfloat16, device="cuda")
    if wo_a:
        outs["y"] = torch.empty(B, S, x["wo_a"].shape[0] * x["wo_a"].shape[2], dtype=torch.bfloat16,
                                device="cuda")
    ws = V.alloc_workspace(cfg)
    V.v4_reset_device_status()
    V.v4_attn_layer_fwd(cfg, xd, outs, ws)
    torch.cuda.synchronize()
    assert V.v4_get_device_status() == 0
    iqp = V.v4_indexer_prep(cfg, x["iq"], xd["inv_freq"], torch.empty_like(x["iq"])) if K else None
    return x, f, outs, iqp


def test_long_context_csa_layer_sampled_rows():
    """S=65536: rows up to 16384 visible entries, several score tiles and
    top-k passes beyond the S=16384 case; the rows around each power of two
    of the entry count and the last row are always sampled."""
    p = SI.preset("csa_bf16_16k", S=65536)
    x, f, outs, iqp = _layer(p, seed=13)
    S = p["S"]
    rows = np.unique(np.concatenate([np.linspace(0, S - 1, 120).round().astype(int),
                                     [0, 1, 127, 128, 2047, 2048, 2051, 8191, 16383, 16384, 32767, 32768,
                                      65531, S - 1]]))
    check_layer_sampled_rows(p, x, outs, rows, f, iqp)
    del x, outs, iqp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", ["csa", "hca", "swa"])
def test_stack_layer_b2_sampled_rows(kind):
    """One layer of each kind of the 43-layer stack as the benchmark runs it
    (B=2, S=16384, with the grouped output projection), both batch elements."""
    name = {"swa": "swa_bf16_16k", "csa": "csa_bf16_16k", "hca": "hca_bf16_16k"}[kind]
    p = SI.preset(name, B=2)
    x, f, outs, iqp = _layer(p, seed=21, wo_a=True)
    S = p["S"]
    rows = np.unique(np.concatenate([np.linspace(0, S - 1, 60).round().astype(int),
                                     [0, 1, 127, 128, 2047, 2048, S - 1]]))
    for b in range(p["B"]):
        check_layer_sampled_rows(p, x, outs, rows, f, iqp, b=b)
    del x, outs, iqp
    torch.cuda.empty_cache()
