"""The workspace-free attention entry point against the workspace one.

v4_sparse_mqa_fwd_noalloc serves callers that cannot allocate device memory
where they run the attention; it keeps its scratch in a library-owned device
array.  Its results must match v4_sparse_mqa_fwd on the same inputs, on two
calls in a row (the second call reuses the array the first one left behind).
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


@pytest.mark.parametrize("mode,base,over", [
    ("csa", "csa_bf16_4k", dict(S=2048, q_mode="direct")),
    ("hca", "hca_bf16_16k", dict(S=3000, q_mode="direct")),
    ("csa_tiny_f32", "tiny_csa_f32", dict()),
])
def test_noalloc_matches_workspace_entry_point(mode, base, over):
    from sparse_compressed_attention_gb300 import build
    build.build()
    lib = V.lib()
    p = SI.preset(base, **over)
    sel = "csa" if mode.startswith("csa") else "hca"
    x, f, ent, idx = _inputs(p, sel, seed=3)
    cfg = V.config_from_preset(p, K=p["K"] if sel == "csa" else 0)
    B, S, H = p["B"], p["S"], p["H"]
    o_ref = torch.empty_like(x["q"])
    l_ref = torch.empty(B, S, H, device="cuda")
    V.v4_sparse_mqa_fwd(cfg, x["q"], x["kv"], ent, idx, x["sink"], f, o_ref, l_ref, V.alloc_workspace(cfg))
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    tol = 1e-5 if p["dtype"] == "f32" else 1e-2
    for call in range(2):
        o = torch.full_like(x["q"], float("nan"))
        lse = torch.full((B, S, H), float("nan"), device="cuda")
        st = lib.v4_sparse_mqa_fwd_noalloc(C.byref(cfg), _ptr(x["q"]), _ptr(x["kv"]), _ptr(ent), _ptr(idx),
                                           _ptr(x["sink"]), _ptr(f), _ptr(o), _ptr(lse), stream)
        assert st == 0, lib.v4_last_error().decode()
        torch.cuda.synchronize()
        assert rel_l2(np64(o), np64(o_ref)) < tol, call
        assert torch.isfinite(lse).all()
        assert np.max(np.abs(np64(lse) - np64(l_ref))) < 1e-3, call
    assert V.v4_get_device_status() == 0


def test_noalloc_rejects_problems_above_its_limit():
    lib = V.lib()
    p = SI.preset("hca_bf16_16k", S=8200)
    cfg = V.config_from_preset(p)
    st = lib.v4_sparse_mqa_fwd_noalloc(C.byref(cfg), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), None, None,
                                       C.c_void_p(16), C.c_void_p(16), None, None)
    assert st == V._lib.V4_ERR_INVALID_ARG
    assert "8192" in lib.v4_last_error().decode()
