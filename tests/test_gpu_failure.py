"""Device-side failure detection without a GPU fault.

Every wait of the tensor-core kernels is bounded: when it runs out, the
kernel records V4_ERR_TIMEOUT in the sticky status word and returns, so the
context stays usable.  The self-test kernel makes such a wait run out (a
barrier nothing completes, a 2 ms limit, no tensor-core or TMA work in
flight); the host reads the status, clears it and runs attention again.
"""
import time

import numpy as np
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from oracle import v4_oracle as O
from tests.helpers import inv_freq_for, np64, rel_l2

pytestmark = pytest.mark.gpu


def _attention_ok():
    p = SI.preset("hca_bf16_16k", S=640, q_mode="direct")
    x = SI.make_layer_inputs(p, "cuda", seed=9)
    f = inv_freq_for(p)
    ent = SI.make_entries(p, "cuda")
    cfg = V.config_from_preset(p)
    o = torch.empty_like(x["q"])
    V.v4_sparse_mqa_fwd(cfg, x["q"], x["kv"], ent, None, None, torch.from_numpy(f).cuda(), o, None,
                        V.alloc_workspace(cfg))
    torch.cuda.synchronize()
    ref, _ = O.sparse_mqa(np64(x["q"]), np64(x["kv"]), np64(ent), None, None, f, p["ratio"], p["W"],
                          store_bf16=True)
    return rel_l2(np64(o), ref)


def test_bounded_wait_times_out_and_the_context_survives():
    from sparse_compressed_attention_gb300 import build
    build.build()
    V.v4_reset_device_status()
    torch.cuda.synchronize()
    assert V.v4_get_device_status() == 0
    t0 = time.time()
    V.v4_selftest_wait_timeout(2000)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert V.v4_get_device_status() == V._lib.V4_ERR_TIMEOUT
    assert elapsed < 1.0                      # the 2 ms limit, not a hang
    V.v4_reset_device_status()
    assert V.v4_get_device_status() == 0
    assert _attention_ok() < 1e-2             # the context still computes
    assert V.v4_get_device_status() == 0


def test_selftest_rejects_bad_limits():
    with pytest.raises(V.V4Error, match="limit_us"):
        V.v4_selftest_wait_timeout(0)
    with pytest.raises(V.V4Error, match="limit_us"):
        V.v4_selftest_wait_timeout(10 ** 7)
