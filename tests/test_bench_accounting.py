"""The benchmark's algorithmic work counts against the oracle's definitions
(CPU only): the keys every query attends to (selected or visible entries
plus its window), the indexer's visible (query, entry) pairs, and the FLOP
totals the roofline fractions divide by at the benchmark sizes."""
import numpy as np
import pytest

import bench
import seeded_inputs as SI
from oracle import v4_oracle as O


@pytest.mark.parametrize("S,r,K,W", [(300, 4, 16, 16), (1000, 4, 64, 128), (700, 128, 0, 128), (257, 0, 0, 37),
                                     (90, 1, 0, -1), (50, 4, 0, 0)])
def test_attention_keys_match_the_oracle(S, r, K, W):
    brute = sum(O.keys_read(t, r, W, K) for t in range(S))
    assert bench.attention_keys_total(S, r, K, W) == brute


def test_indexer_pairs_match_visibility():
    p = SI.preset("csa_bf16_4k", S=999)
    brute = sum(min(O.n_visible(t, p["ratio"]), p["S"] // p["ratio"]) for t in range(p["S"]))
    assert bench.layer_work(p)["idx_pairs"] == brute


def test_flop_totals_at_the_benchmark_sizes():
    csa = bench.layer_work(SI.preset("csa_bf16_16k"))
    hca = bench.layer_work(SI.preset("hca_bf16_16k"))
    H, D = 64, 512
    assert csa["attn_flops"] == 4.0 * H * D * csa["attn_keys"]
    assert abs(csa["attn_flops"] / 1e12 - 1.3045) < 1e-3        # 1.305 TFLOP per CSA attention launch
    assert abs(hca["attn_flops"] / 1e12 - 0.4092) < 1e-3
    assert abs(csa["idx_flops"] / 1e12 - 0.5497) < 1e-3         # 0.550 TFLOP per indexer launch
    assert csa["attn_bytes"] == hca["attn_bytes"] == 2 * 16384 * H * D * 2


def test_layer_rooflines_at_the_benchmark_sizes():
    """The CSA layer is tensor-bound and the HCA layer HBM-bound at S=16384
    (q + o dominate HCA's bytes: 2.15 GB against 0.41 TFLOP); a layer that
    runs exactly at its bound reads 1.0."""
    peaks = {"bf16": 1932.6, "hbm": 6779.0}
    csa = bench.layer_work(SI.preset("csa_bf16_16k"))
    hca = bench.layer_work(SI.preset("hca_bf16_16k"))
    S, H, D, Hi, Di, K = 16384, 64, 512, 64, 128, 512
    # inputs read once and outputs written once; CSA adds its indexer's
    assert hca["layer_bytes"] == 2 * S * H * D * 2 + S * D * 2 + 2 * S * D * 2
    assert csa["layer_bytes"] == (2 * S * H * D * 2 + S * D * 2 + 2 * S * 2 * D * 2
                                  + S * Hi * Di * 2 + 2 * S * 2 * Di * 2 + S * Hi * 4 + S * K * 4)
    rc = bench.layer_roofline("csa", csa, 10.0, peaks)
    rh = bench.layer_roofline("hca", hca, 10.0, peaks)
    assert rc["bound"] == "tensor" and rh["bound"] == "hbm"
    assert abs(rc["bound_ms"] - csa["layer_flops"] / 1932.6e12 * 1e3) < 1e-4
    at_bound = bench.layer_roofline("hca", hca, hca["layer_bytes"] / 6779e9 * 1e3, peaks)
    assert abs(at_bound["frac"] - 1.0) < 1e-3


def test_row_chunk_work_adds_up_to_the_whole_sequence():
    """The work of a rank's query rows: the chunks of a split add up to the
    whole layer's FLOPs (attention keys and indexer pairs) and q + o bytes."""
    from sparse_compressed_attention_gb300 import rows as R
    for name in ("csa_bf16_16k", "hca_bf16_16k"):
        p = SI.preset(name, S=3000)
        whole = bench.layer_work(p)
        cost = R.layer_cost(p["ratio"], p["K"], p["W"], tile=128)
        parts = [bench.layer_work(p, R.contiguous_chunks(p["S"], 4, r, cost)) for r in range(4)]
        for key in ("attn_flops", "attn_bytes", "idx_flops", "attn_keys", "idx_pairs"):
            assert sum(w[key] for w in parts) == whole[key], (name, key)
        # bench's rank chunks: whole sequence at N=1, the contiguous split otherwise
        assert bench.rank_chunks(p, 1, 0) == [(0, p["S"])]
        assert sum(b - a for r in range(3) for a, b in bench.rank_chunks(p, 3, r)) == p["S"]


def test_stack_mix_and_its_roofline_inputs():
    """The 43-layer stack the bench measures: 2 window-only + 21 CSA + 20 HCA
    layers in the Flash order, and the per-kind counts its roofline sums."""
    assert bench.STACK_ORDER[:2] == ["swa", "swa"] and bench.STACK_ORDER[-1] == "csa"
    assert {k: bench.STACK_ORDER.count(k) for k in set(bench.STACK_ORDER)} == bench.STACK_COUNTS
    assert sum(bench.STACK_COUNTS.values()) == 43
    ratios = [{"swa": 0, "csa": 4, "hca": 128}[k] for k in bench.STACK_ORDER]
    assert ratios == SI.flash_layer_ratios()
