"""The seeded input generators (CPU): shapes, dtypes, the stated
distributions' defining properties, and that a seed fixes every draw."""
import torch

import seeded_inputs as SI


def _rms(x):
    return x.float().pow(2).mean(dim=-1).sqrt()


def test_indexer_operands():
    p = SI.preset("csa_bf16_4k", S=300, B=2)
    iqp, ikey, w = SI.make_indexer_operands(p, "cpu", seed=5)
    assert iqp.shape == (2, 300, p["Hi"], p["Di"]) and iqp.dtype == torch.bfloat16
    assert ikey.shape == (2, 300 // p["ratio"], p["Di"]) and ikey.dtype == torch.bfloat16
    assert w.shape == (2, 300, p["Hi"]) and w.dtype == torch.float32
    # unit-RMS rows up to the bf16 rounding of their elements
    assert torch.allclose(_rms(iqp), torch.ones(1), atol=1e-2)
    assert torch.allclose(_rms(ikey), torch.ones(1), atol=1e-2)
    again = SI.make_indexer_operands(p, "cpu", seed=5)
    assert all(torch.equal(a, b) for a, b in zip((iqp, ikey, w), again))
    other = SI.make_indexer_operands(p, "cpu", seed=6)
    assert not torch.equal(iqp, other[0])


def test_layer_inputs_are_seeded_and_unit_rms():
    p = SI.preset("tiny_csa_f32")
    x = SI.make_layer_inputs(p, "cpu", seed=3)
    y = SI.make_layer_inputs(p, "cpu", seed=3)
    for k, v in x.items():
        if v is not None:
            assert torch.equal(v, y[k]), k
    for k in ("q", "kv", "ckv", "cscore", "ickv", "icscore", "iq"):
        assert torch.allclose(_rms(x[k]), torch.ones(1), atol=1e-5), k


def test_random_selections_are_valid():
    idx = SI.random_topk_indices(2, 90, 4, 8, "cpu", seed=2)
    for b in range(2):
        for t in range(90):
            row = idx[b, t]
            sel = row[row >= 0]
            nv = (t + 1) // 4
            assert len(sel) == min(8, nv)
            assert len(set(sel.tolist())) == len(sel) and (sel < nv).all()
