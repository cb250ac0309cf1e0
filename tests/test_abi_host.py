"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, validates arguments before touching a GPU, and builds the same RoPE
table as the oracle.  No kernel runs here."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

import seeded_inputs as SI
from oracle import v4_oracle as O
from sparse_compressed_attention_gb300 import _lib as L
from sparse_compressed_attention_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "v4attn.h")).read()
    return sorted(set(re.findall(r"^\s*(?:v4_status|const char\*|uint64_t|int32_t)\s+(v4_\w+)\s*\(", text, re.M)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(L.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (v4_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


@pytest.mark.parametrize("theta,R,yarn,olen", [(40000.0, 64, 16.0, 4096), (10000.0, 64, 1.0, 0),
                                               (40000.0, 16, 1.0, 0), (160000.0, 128, 40.0, 4096)])
def test_inv_freq_table_matches_oracle(lib, theta, R, yarn, olen):
    got = L.v4_rope_inv_freq(theta, R, yarn, olen, 32.0, 1.0).numpy()
    ref = O.make_inv_freq(theta, R, yarn, olen, 32.0, 1.0)
    ulps = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1


def test_workspace_size_covers_layer_buffers(lib):
    p = SI.preset("csa_bf16_16k")
    cfg = L.config_from_preset(p)
    n = L.v4_workspace_size(cfg)
    S, N = 16384, 4096
    need = S * 512 * 2 + N * 512 * 2 + N * 128 * 2 + S * 64 * 128 * 2 + S * N * 4 + S * 512 * 4
    assert n >= need
    hca = L.v4_workspace_size(L.config_from_preset(SI.preset("hca_bf16_16k")))
    assert hca < n


def _status(fn, *args):
    return fn(*args)


@pytest.mark.parametrize("field,value,msg", [
    ("head_dim", 40, "head_dim"), ("rope_dim", 12, "rope_dim"), ("ratio", -1, "ratio"),
    ("overlap", 2, "overlap"), ("window", -2, "window"), ("topk", -1, "topk"),
    ("idx_dim", 96, "idx_dim"), ("dtype", 7, "dtype"), ("batch", 0, "batch"),
    ("indexer_fp8", 2, "indexer_fp8")])
def test_invalid_config_is_rejected_on_host(lib, field, value, msg):
    cfg = L.config_from_preset(SI.preset("csa_bf16_4k"))
    setattr(cfg, field, value)
    n = C.c_size_t(0)
    st = lib.v4_workspace_size(C.byref(cfg), C.byref(n))
    assert st == L.V4_ERR_INVALID_ARG
    assert msg in lib.v4_last_error().decode()


def test_null_and_misaligned_pointers_are_rejected(lib):
    cfg = L.config_from_preset(SI.preset("csa_bf16_4k"))
    st = lib.v4_compress(C.byref(cfg), None, 16, 16, None, 16, 512, 0, 16, None)
    assert st == L.V4_ERR_INVALID_ARG and "ckv" in lib.v4_last_error().decode()
    st = lib.v4_compress(C.byref(cfg), 24, 16, 16, None, 16, 512, 0, 16, None)
    assert st == L.V4_ERR_INVALID_ARG and "aligned" in lib.v4_last_error().decode()
    st = lib.v4_compress(C.byref(cfg), 16, 16, 16, None, 16, 384, 1, 16, None)
    assert st == L.V4_ERR_INVALID_ARG and "Hadamard" in lib.v4_last_error().decode()


def test_workspace_too_small_is_rejected(lib):
    cfg = L.config_from_preset(SI.preset("csa_bf16_4k"))
    st = lib.v4_indexer_topk(C.byref(cfg), 16, 0, 16, 16, 16, 16, None, 256, 1024, None)
    assert st == L.V4_ERR_WORKSPACE and "needed" in lib.v4_last_error().decode()


def test_topk_without_ratio_is_rejected(lib):
    cfg = L.make_config(1, 64, 4, 64, 16, ratio=0, topk=8, Hi=2, Di=32)
    st = lib.v4_indexer_topk(C.byref(cfg), 16, 0, 16, 16, 16, 16, None, 256, 1 << 20, None)
    assert st == L.V4_ERR_INVALID_ARG and "ratio" in lib.v4_last_error().decode()


def test_e4m3_indexer_host_checks(lib):
    # the workspace trades the bf16 prepared queries for the codes and scales
    # of both operands
    p = SI.preset("csa_bf16_4k")
    n0 = L.v4_workspace_size(L.config_from_preset(p))
    n1 = L.v4_workspace_size(L.config_from_preset(p, indexer_fp8=1))
    S, N = p["S"], p["S"] // p["ratio"]
    assert n1 >= n0 - S * 64 * 128 * 2 + S * 64 * 128 + S * 64 * 4 + N * 128 + N * 4
    assert n1 < n0
    # shapes outside the tensor-core indexer are refused before any launch
    cfg = L.config_from_preset(SI.preset("tiny_csa_f32"), indexer_fp8=1)
    st = lib.v4_indexer_topk_e4m3(C.byref(cfg), 16, 16, 16, 16, 16, 16, None, 256, 1 << 20, None)
    assert st == L.V4_ERR_UNSUPPORTED and "E4M3" in lib.v4_last_error().decode()
    st = lib.v4_indexer_topk(C.byref(cfg), 16, 0, 16, 16, 16, 16, None, 256, 1 << 20, None)
    assert st == L.V4_ERR_UNSUPPORTED and "E4M3" in lib.v4_last_error().decode()
    cfg = L.config_from_preset(p, indexer_fp8=1, path=L.V4_PATH_SIMT)
    st = lib.v4_indexer_topk(C.byref(cfg), 16, 0, 16, 16, 16, 16, None, 256, 1 << 30, None)
    assert st == L.V4_ERR_UNSUPPORTED
    # the quantiser's own argument checks
    st = lib.v4_quantize_e4m3(16, 4, 100, 16, 16, None)
    assert st == L.V4_ERR_INVALID_ARG and "dim" in lib.v4_last_error().decode()
    st = lib.v4_quantize_e4m3(None, 4, 128, 16, 16, None)
    assert st == L.V4_ERR_INVALID_ARG and "x" in lib.v4_last_error().decode()
    assert lib.v4_quantize_e4m3(None, 0, 128, None, None, None) == L.V4_OK


def test_q_projection_host_checks(lib):
    cfg = L.config_from_preset(SI.preset("tiny_csa_f32"))
    st = lib.v4_q_proj(C.byref(cfg), 16, 1024, 16, 1, None, None, 16, None, None)
    assert st == L.V4_ERR_UNSUPPORTED and "bf16" in lib.v4_last_error().decode()
    cfg = L.config_from_preset(SI.preset("csa_bf16_4k"))
    st = lib.v4_q_proj(C.byref(cfg), 16, 1000, 16, 1, None, None, 16, None, None)
    assert st == L.V4_ERR_UNSUPPORTED
    st = lib.v4_q_proj(C.byref(cfg), 16, 1024, 16, 2, None, None, 16, None, None)
    assert st == L.V4_ERR_INVALID_ARG and "q_norm" in lib.v4_last_error().decode()
    st = lib.v4_q_proj(C.byref(cfg), 16, 1024, 16, 1, None, 16, 16, None, None)
    assert st == L.V4_ERR_INVALID_ARG and "iq" in lib.v4_last_error().decode()


def test_error_text_is_per_thread(lib):
    import threading
    cfg = L.config_from_preset(SI.preset("csa_bf16_4k"))
    cfg.head_dim = 40
    n = C.c_size_t(0)
    lib.v4_workspace_size(C.byref(cfg), C.byref(n))
    seen = []
    th = threading.Thread(target=lambda: seen.append(lib.v4_last_error().decode()))
    th.start()
    th.join()
    assert seen == [""]
    assert "head_dim" in lib.v4_last_error().decode()


def test_row_slice_argument_checks(lib):
    # q_begin must name a query position; the backward and the distillation
    # target take whole sequences only (both refused before any GPU work)
    p = SI.preset("hca_bf16_16k", S=256, q_mode="direct")
    with pytest.raises(L.V4Error, match="q_begin"):
        L.v4_workspace_size(L.config_from_preset(p, q_begin=256))
    with pytest.raises(L.V4Error, match="q_begin"):
        L.v4_workspace_size(L.config_from_preset(p, q_begin=-1))
    cfg = L.config_from_preset(p, q_begin=64)
    st = lib.v4_sparse_mqa_bwd(C.byref(cfg), *([None] * 14), 0, None)
    assert st == L.V4_ERR_UNSUPPORTED and "q_begin" in lib.v4_last_error().decode()
    csa = L.config_from_preset(SI.preset("csa_bf16_4k", S=256, q_mode="direct"), q_begin=8)
    st = lib.v4_indexer_kl_target(C.byref(csa), *([None] * 9), None, 0, None)
    assert st == L.V4_ERR_UNSUPPORTED and "q_begin" in lib.v4_last_error().decode()


def test_workspace_of_a_row_slice_scales_with_its_rows(lib):
    p = SI.preset("csa_bf16_16k")
    whole = L.v4_workspace_size(L.config_from_preset(p))
    tail = L.v4_workspace_size(L.config_from_preset(p, q_begin=12288))
    # the prepared queries, scores and selection shrink to a quarter of the rows
    S, N = 16384, 4096
    row_bytes = 64 * 128 * 2 + N * 4 + 512 * 4
    assert whole - tail >= 0.75 * S * row_bytes - 4096
