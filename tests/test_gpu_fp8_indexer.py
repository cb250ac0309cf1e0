"""Opt-in E4M3 indexer on the GPU against the oracle.

Stage by stage: the quantiser is bit-exact (codes and float32 scales) on
bf16 rows made by the oracle (ragged row counts, zero rows, a dominant value,
subnormal codes, every supported width); the E4M3 scores and top-k, fed
codes and scales made by the oracle, select the oracle's sets outside the
fp32 tie band.  End to end, the layer with ``indexer_fp8 = 1`` follows the
oracle's E4M3 pipeline (its own entries, keys, prepared queries, quantiser
and selection): >= 99.5% of selected entries agree and the output is within
1e-2 relative L2.  How much E4M3 changes the selection against the exact
(bf16 operands, fp64 scoring) one is measured on the same rows and bounded
loosely: it is a property of the quantisation, not a parity claim.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
import sparse_compressed_attention_gb300 as V
from oracle import v4_oracle as O
from tests.helpers import check_topk_rows, inv_freq_for, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_compressed_attention_gb300 import build
    build.build()


def _to_codes(vals):
    """E4M3 values (float64, exactly representable) -> uint8 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(vals)).float().to(torch.float8_e4m3fn).view(torch.uint8).cuda()


def _from_codes(t):
    return t.view(torch.float8_e4m3fn).float().cpu().numpy().astype(np.float64)


def _overlap(a_idx, b_idx):
    agree = total = 0
    for a, b in zip(a_idx.reshape(-1, a_idx.shape[-1]), b_idx.reshape(-1, b_idx.shape[-1])):
        sa, sb = set(a[a >= 0].tolist()), set(b[b >= 0].tolist())
        assert len(sa) == len(sb)
        agree += len(sa & sb)
        total += len(sb)
    return agree / max(1, total)


@pytest.mark.parametrize("rows,dim", [(1, 128), (37, 128), (4099, 128), (300, 256), (65, 512), (9, 1024)])
def test_quantizer_bit_exact(rows, dim):
    rng = np.random.default_rng(rows * 7 + dim)
    x = rng.normal(0, 1, (rows, dim))
    x *= np.exp(rng.normal(0, 3, (rows, 1)))          # row magnitudes over many binades
    if rows > 3:
        x[1] = 0.0
        x[2, 5] = 1e3 * np.abs(x[2]).max()             # one dominant value: most codes subnormal
        x[3] = np.abs(x[3])
    x = O.round_to_bf16(x)
    codes, scales = O.quantize_e4m3_rows(x)
    xd = torch.from_numpy(x).to(torch.bfloat16).cuda()
    gc = torch.empty(rows, dim, dtype=torch.uint8, device="cuda")
    gs = torch.empty(rows, dtype=torch.float32, device="cuda")
    V.v4_quantize_e4m3(xd, gc, gs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_from_codes(gc), codes)
    np.testing.assert_array_equal(gs.cpu().numpy(), scales.astype(np.float32))


def _oracle_operands(p, x, f):
    ikey = O.compress(np64(x["ickv"]), np64(x["icscore"]), np64(x["iape"]), None, f, p["ratio"],
                      p["overlap"], 1e-6, hadamard=True, store_bf16=True)
    iqp = O.indexer_query_prep(np64(x["iq"]), f, store_bf16=True)
    qc, qs = O.quantize_e4m3_rows(iqp)
    kc, ks = O.quantize_e4m3_rows(ikey)
    return ikey, iqp, qc, qs, kc, ks


@pytest.mark.parametrize("name,p", [
    ("s1024", SI.preset("csa_bf16_4k", S=1024, q_mode="direct")),
    ("ragged_b2_k64", SI.preset("csa_bf16_4k", S=777, B=2, K=64, q_mode="direct")),
    ("s3001", SI.preset("csa_bf16_4k", S=3001, q_mode="direct")),
])
def test_e4m3_indexer_topk_stagewise(name, p):
    x = SI.make_layer_inputs(p, "cpu", seed=0)
    f = inv_freq_for(p)
    _, _, qc, qs, kc, ks = _oracle_operands(p, x, f)
    cfg = V.config_from_preset(p, indexer_fp8=1)
    B, S, K = p["B"], p["S"], p["K"]
    idx = torch.empty(B, S, K, dtype=torch.int32, device="cuda")
    isc = torch.empty(B, S, K, dtype=torch.float32, device="cuda")
    V.v4_indexer_topk_e4m3(cfg, _to_codes(qc), torch.from_numpy(qs).float().cuda(), _to_codes(kc),
                           torch.from_numpy(ks).float().cuda(), x["w"].cuda(), idx, isc, V.alloc_workspace(cfg))
    torch.cuda.synchronize()
    assert V.v4_get_device_status() == 0
    gi, gs = idx.cpu().numpy(), isc.cpu().numpy()
    w = np64(x["w"])
    c = O.indexer_scale(p["Hi"], p["Di"])
    qd = qc * qs[..., None]                            # the exact operands both sides score
    kd = kc * ks[..., None]
    swaps = 0
    for b in range(B):
        sc = O.indexer_scores(qd[b:b + 1], kd[b:b + 1], w[b:b + 1], p["ratio"])[0]
        swaps += check_topk_rows(gi[b], sc, qd[b], kd[b], w[b], p["ratio"], K, range(S), c)
        for t in range(S):
            row = gi[b, t]
            kept = row[row >= 0]
            assert np.all(np.diff(kept) > 0)
            if len(kept):
                band = 4 * (p["Di"] + p["Hi"] + 8) * 2.0 ** -24 * (np.abs(w[b, t]) * c) @ (
                    np.abs(qd[b, t]) @ np.abs(kd[b, kept]).T)
                assert np.all(np.abs(gs[b, t, :len(kept)] - sc[t, kept]) <= band + 1e-30)
    assert swaps <= max(2, B * S * K // 10000)


def test_prepared_queries_quantised_by_the_library():
    # v4_indexer_topk with E4M3 on queries the caller prepared (bf16, made by
    # the oracle): the library quantises them with the standalone rule
    p = SI.preset("csa_bf16_4k", S=1500, q_mode="direct")
    x = SI.make_layer_inputs(p, "cpu", seed=2)
    f = inv_freq_for(p)
    ikey, iqp, qc, qs, kc, ks = _oracle_operands(p, x, f)
    cfg = V.config_from_preset(p, indexer_fp8=1)
    B, S, K = p["B"], p["S"], p["K"]
    idx = torch.empty(B, S, K, dtype=torch.int32, device="cuda")
    V.v4_indexer_topk(cfg, torch.from_numpy(iqp).to(torch.bfloat16).cuda(), 1,
                      torch.from_numpy(ikey).to(torch.bfloat16).cuda(), x["w"].cuda(),
                      torch.from_numpy(f).cuda(), idx, None, V.alloc_workspace(cfg))
    torch.cuda.synchronize()
    sel = O.indexer_topk_e4m3(qc, qs, kc, ks, np64(x["w"]), p["ratio"], K)["idx"]
    assert _overlap(idx.cpu().numpy(), sel) >= 0.995


def _layer(p, x, f, fp8):
    xd = dict(to_dev(x), inv_freq=torch.from_numpy(f).cuda())
    cfg = V.config_from_preset(p, indexer_fp8=fp8)
    B, S, H, K = p["B"], p["S"], p["H"], p["K"]
    outs = {"o": torch.empty_like(xd["q"]), "lse": torch.empty(B, S, H, device="cuda"),
            "idx": torch.empty(B, S, K, dtype=torch.int32, device="cuda")}
    V.v4_reset_device_status()
    V.v4_attn_layer_fwd(cfg, xd, outs, V.alloc_workspace(cfg))
    torch.cuda.synchronize()
    assert V.v4_get_device_status() == 0
    return outs


@pytest.mark.parametrize("name,p", [
    ("s1024", SI.preset("csa_bf16_4k", S=1024, q_mode="direct")),
    ("b2_s700_k128", SI.preset("csa_bf16_4k", S=700, B=2, K=128, q_mode="direct")),
])
def test_layer_e4m3_end_to_end(name, p):
    x = SI.make_layer_inputs(p, "cpu", seed=0)
    f = inv_freq_for(p)
    outs = _layer(p, x, f, 1)
    ikey, _, qc, qs, kc, ks = _oracle_operands(p, x, f)
    sel = O.indexer_topk_e4m3(qc, qs, kc, ks, np64(x["w"]), p["ratio"], p["K"])["idx"]
    g = outs["idx"].cpu().numpy()
    assert _overlap(g, sel) >= 0.995
    ent = O.compress(np64(x["ckv"]), np64(x["cscore"]), np64(x["ape"]), None, f, p["ratio"], p["overlap"],
                     1e-6, store_bf16=True)
    ro, _ = O.sparse_mqa(np64(x["q"]), np64(x["kv"]), ent, sel, None, f, p["ratio"], p["W"], store_bf16=True)
    assert rel_l2(np64(outs["o"]), ro) < 1e-2
    # the measured effect of E4M3 on the selection (against exact scoring)
    exact = O.indexer_topk(np64(x["iq"]), ikey, np64(x["w"]), f, p["ratio"], p["K"], store_bf16=True)["idx"]
    kept = _overlap(sel, exact)
    print("E4M3 keeps %.4f of the exact selection (%s)" % (kept, name))
    assert kept >= 0.8


def test_full_size_e4m3_layer_sampled_rows():
    """The bench's S=16384 CSA layer with the E4M3 indexer, checked on ~510
    sampled rows against the oracle's E4M3 selection and output."""
    p = SI.preset("csa_bf16_16k")
    x = SI.make_layer_inputs(p, "cuda", seed=11)
    f = inv_freq_for(p)
    outs = _layer(p, x, f, 1)
    S, K = p["S"], p["K"]
    rows = np.unique(np.concatenate([np.linspace(0, S - 1, 504).round().astype(int),
                                     [0, 1, 127, 128, 511, 512, 2047, S - 1]]))
    rsel = torch.from_numpy(rows).cuda()
    ikey = O.compress(np64(x["ickv"]), np64(x["icscore"]), np64(x["iape"]), None, f, p["ratio"],
                      p["overlap"], 1e-6, hadamard=True, store_bf16=True)
    iqp = O.indexer_query_prep(np64(x["iq"][:, rsel]), f, store_bf16=True, positions=rows)
    qc, qs = O.quantize_e4m3_rows(iqp)
    kc, ks = O.quantize_e4m3_rows(ikey)
    w_rows = np64(x["w"][:, rsel])
    sel = O.indexer_topk_e4m3(qc, qs, kc, ks, w_rows, p["ratio"], K, rows=rows, rows_only=True)["idx"]
    gi = outs["idx"][:, rsel].cpu().numpy()
    assert _overlap(gi, sel) >= 0.99
    exact = O.indexer_topk(np64(x["iq"][:, rsel]), ikey, w_rows, f, p["ratio"], K, store_bf16=True, rows=rows,
                           rows_only=True)["idx"]
    kept = _overlap(sel, exact)
    print("E4M3 keeps %.4f of the exact top-%d at S=%d" % (kept, K, S))
    assert kept >= 0.8
    ent = O.compress(np64(x["ckv"]), np64(x["cscore"]), np64(x["ape"]), None, f, p["ratio"], p["overlap"],
                     1e-6, store_bf16=True)
    ro, _ = O.sparse_mqa(np64(x["q"][:, rsel]), np64(x["kv"]), ent, sel, None, f, p["ratio"], p["W"],
                         store_bf16=True, rows=rows, rows_only=True)
    assert rel_l2(np64(outs["o"][:, rsel]), ro) < 1e-2
