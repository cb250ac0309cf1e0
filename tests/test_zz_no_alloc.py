"""The workspace-free attention entry point against the workspace one.

v4_sparse_mqa_fwd_noalloc serves callers that cannot allocate device memory
where they run the attention; it keeps its scratch in a library-owned device
array.  Its results must match v4_sparse_mqa_fwd on the same inputs, on calls in a
row with a different problem in between (each call starts from whatever the
previous one left in the array).
"""
import ctypes as C

import numpy as np
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from oracle import v4_oracle as O
from tests.helpers import inv_freq_for, np64, rel_l2

pytestmark = pytest.mark.gpu


def _inputs(p, mode, seed):
    x = SI.make_layer_inputs(p, "cuda", seed=seed, sink=True)
    f = torch.from_numpy(inv_freq_for(p)).cuda()
    ent = idx = None
    if p["ratio"] > 0:
        e = O.compress(np64(x["ckv"]), np64(x["cscore"]), np64(x["ape"]), None, inv_freq_for(p), p["ratio"],
                       p["overlap"], 1e-6, store_bf16=True)
        ent = torch.from_numpy(e).to(x["q"].dtype).cuda()
    if mode == "csa":
        idx = SI.random_topk_indices(p["B"], p["S"], p["ratio"], p["K"], "cuda", seed=seed + 1)
    return x, f, ent, idx


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _problem(mode, base, over, seed):
    p = SI.preset(base, **over)
    sel = "csa" if mode.startswith("csa") else "hca"
    x, f, ent, idx = _inputs(p, sel, seed=seed)
    cfg = V.config_from_preset(p, K=p["K"] if sel == "csa" else 0)
    B, S, H = p["B"], p["S"], p["H"]
    o_ref = torch.empty_like(x["q"])
    l_ref = torch.empty(B, S, H, device="cuda")
    V.v4_sparse_mqa_fwd(cfg, x["q"], x["kv"], ent, idx, x["sink"], f, o_ref, l_ref, V.alloc_workspace(cfg))
    return dict(p=p, x=x, f=f, ent=ent, idx=idx, cfg=cfg, o_ref=o_ref, l_ref=l_ref)


def _call_and_check(lib, pr, tag):
    p, x = pr["p"], pr["x"]
    B, S, H = p["B"], p["S"], p["H"]
    o = torch.full_like(x["q"], float("nan"))
    lse = torch.full((B, S, H), float("nan"), device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.v4_sparse_mqa_fwd_noalloc(C.byref(pr["cfg"]), _ptr(x["q"]), _ptr(x["kv"]), _ptr(pr["ent"]),
                                       _ptr(pr["idx"]), _ptr(x["sink"]), _ptr(pr["f"]), _ptr(o), _ptr(lse), stream)
    assert st == 0, lib.v4_last_error().decode()
    torch.cuda.synchronize()
    tol = 1e-5 if p["dtype"] == "f32" else 1e-2
    assert rel_l2(np64(o), np64(pr["o_ref"])) < tol, tag
    assert torch.isfinite(lse).all(), tag
    assert np.max(np.abs(np64(lse) - np64(pr["l_ref"]))) < 1e-3, tag


@pytest.mark.parametrize("mode,base,over,other", [
    ("csa", "csa_bf16_4k", dict(S=2048, q_mode="direct"), ("hca", "hca_bf16_16k", dict(S=8000, q_mode="direct"))),
    ("hca", "hca_bf16_16k", dict(S=3000, q_mode="direct"), ("csa", "csa_bf16_4k", dict(S=6000, q_mode="direct"))),
    ("csa_tiny_f32", "tiny_csa_f32", dict(), ("csa_tiny_f32", "tiny_csa_f32", dict(S=200))),
])
def test_noalloc_matches_workspace_entry_point(mode, base, over, other):
    """Three calls in a row, each checked against v4_sparse_mqa_fwd: the
    problem, a different and larger one (which leaves other contents in the
    shared array), then the first problem again."""
    from sparse_compressed_attention_gb300 import build
    build.build()
    lib = V.lib()
    a = _problem(mode, base, over, seed=3)
    b = _problem(*other, seed=7)
    _call_and_check(lib, a, "first call")
    _call_and_check(lib, b, "different problem")
    _call_and_check(lib, a, "first problem again")
    assert V.v4_get_device_status() == 0


def test_noalloc_rejects_problems_above_its_limit():
    lib = V.lib()
    p = SI.preset("hca_bf16_16k", S=8200)
    cfg = V.config_from_preset(p)
    st = lib.v4_sparse_mqa_fwd_noalloc(C.byref(cfg), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), None, None,
                                       C.c_void_p(16), C.c_void_p(16), None, None)
    assert st == V._lib.V4_ERR_INVALID_ARG
    assert "8192" in lib.v4_last_error().decode()
