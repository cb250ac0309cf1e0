"""Seeded synthetic inputs for the compressed-attention forward and backward.

Shared by the tests, ``bench.py`` and the callers of the CPU oracle.  It holds
no step of the attention method: only workload shapes, random draws in a fixed
order, and the unit-RMS scaling that gives the input rows the distribution the
workloads name ("activations RMSNorm(N(0,1))").

The workloads follow the DeepSeek-V4-Flash shapes of the blog "Enabling
DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs with Primus" (section
"The DeepSeek-V4-Flash architecture": 64 query heads, one 512-d K=V latent,
rank-1024 query path, 8 output groups of 1024; section "Three attention types":
ratio 4 with overlapping groups, ratio 128, top-512, 128-token window).
"""
from __future__ import annotations

import torch

# name -> shape and distribution parameters
PRESETS = {
    # Tiny CSA forward in fp32 (parity at 1e-5)
    "tiny_csa_f32": dict(B=1, S=256, H=4, D=64, R=16, theta=40000.0, yarn=1.0,
                         ratio=4, overlap=1, Hi=2, Di=32, K=16, W=16,
                         dtype="f32", ape_std=0.1, q_mode="direct"),
    # CSA layer, bf16, S=4096
    "csa_bf16_4k": dict(B=1, S=4096, H=64, D=512, R=64, theta=40000.0, yarn=16.0,
                        ratio=4, overlap=1, Hi=64, Di=128, K=512, W=128,
                        dtype="bf16", ape_std=0.02, q_mode="lowrank"),
    # CSA layer, bf16, S=16384
    "csa_bf16_16k": dict(B=1, S=16384, H=64, D=512, R=64, theta=40000.0, yarn=16.0,
                         ratio=4, overlap=1, Hi=64, Di=128, K=512, W=128,
                         dtype="bf16", ape_std=0.02, q_mode="lowrank"),
    # HCA layer, bf16, S=16384 (no indexer)
    "hca_bf16_16k": dict(B=1, S=16384, H=64, D=512, R=64, theta=40000.0, yarn=16.0,
                         ratio=128, overlap=0, Hi=64, Di=128, K=0, W=128,
                         dtype="bf16", ape_std=0.02, q_mode="lowrank"),
    # Long-context CSA, bf16, S=65536
    "csa_bf16_64k": dict(B=1, S=65536, H=64, D=512, R=64, theta=40000.0, yarn=16.0,
                         ratio=4, overlap=1, Hi=64, Di=128, K=512, W=128,
                         dtype="bf16", ape_std=0.02, q_mode="lowrank"),
    # Window-only layer (the first two layers of the stack)
    "swa_bf16_16k": dict(B=1, S=16384, H=64, D=512, R=64, theta=10000.0, yarn=1.0,
                         ratio=0, overlap=0, Hi=64, Di=128, K=0, W=128,
                         dtype="bf16", ape_std=0.02, q_mode="lowrank"),
}

# YaRN setting assumed for the compressed layers: the pages give theta 40000
# and factor 16 but not the original length or the ramp bounds.
YARN_ORIGINAL_LEN = 4096
YARN_BETA_FAST = 32.0
YARN_BETA_SLOW = 1.0

Q_RANK = 1024          # low-rank query path
O_GROUPS = 8           # grouped output projection
O_RANK = 1024


def preset(name, **over):
    p = dict(PRESETS[name])
    p.update(over)
    return p


def flash_layer_ratios():
    """Compression ratio of each of the 43 decoder layers of V4-Flash.

    Two window-only layers, then CSA (4) and HCA (128) alternating, starting
    and ending with CSA: 21 CSA + 20 HCA.
    """
    return [0, 0] + [4 if i % 2 == 0 else 128 for i in range(41)]


def torch_dtype(p):
    return torch.float32 if p["dtype"] == "f32" else torch.bfloat16


def _normal(shape, gen, device, std=1.0):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32) * std


def _unit_rms(x):
    return x / x.pow(2).mean(dim=-1, keepdim=True).sqrt()


def make_layer_inputs(p, device="cpu", seed=0, sink=False, wo_a=False):
    """Draw every input of one layer, in a fixed order, on ``device``.

    Activations (kv, pooling projections and scores, indexer projections) are
    unit-RMS rows of N(0,1); ``ape`` ~ N(0, ape_std); indexer weights
    w ~ N(0,1); norm weights are ones.  With q_mode "lowrank" the queries come
    from the rank-1024 path: qlat = unit-RMS N(0,1) [B,S,1024], q = per-head
    unit-RMS(qlat @ Wq), iq = qlat @ Wiq with Wq, Wiq ~ N(0, 0.02).
    Tensors a layer does not use (pooling inputs without compression, indexer
    inputs without selection) are not drawn.  Returns a dict of tensors;
    activations in the preset's storage dtype, parameters (ape, norm weights,
    w, sink) in float32.
    """
    B, S, H, D = p["B"], p["S"], p["H"], p["D"]
    Hi, Di, r, ov = p["Hi"], p["Di"], p["ratio"], p["overlap"]
    dt = torch_dtype(p)
    sel = p["K"] > 0 and r > 0
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = {}
    if p["q_mode"] == "lowrank":
        qlat = _unit_rms(_normal((B, S, Q_RANK), g, device))
        wq = _normal((Q_RANK, H * D), g, device, 0.02)
        q = (qlat @ wq).view(B, S, H, D)
        x["q"] = _unit_rms(q).to(dt)
        del q, wq
        if sel:
            wiq = _normal((Q_RANK, Hi * Di), g, device, 0.02)
            x["iq"] = (qlat @ wiq).view(B, S, Hi, Di).to(dt)
            del wiq
        del qlat
    else:
        x["q"] = _unit_rms(_normal((B, S, H, D), g, device)).to(dt)
        if sel:
            x["iq"] = _unit_rms(_normal((B, S, Hi, Di), g, device)).to(dt)
    x["kv"] = _unit_rms(_normal((B, S, D), g, device)).to(dt)
    G = max(1, (1 + ov) * max(r, 1))
    if r > 0:
        x["ckv"] = _unit_rms(_normal((B, S, 1 + ov, D), g, device)).to(dt)
        x["cscore"] = _unit_rms(_normal((B, S, 1 + ov, D), g, device)).to(dt)
        x["ape"] = _normal((G, D), g, device, p["ape_std"])
        x["norm_w"] = torch.ones(D, device=device)
    if sel:
        x["ickv"] = _unit_rms(_normal((B, S, 1 + ov, Di), g, device)).to(dt)
        x["icscore"] = _unit_rms(_normal((B, S, 1 + ov, Di), g, device)).to(dt)
        x["iape"] = _normal((G, Di), g, device, p["ape_std"])
        x["w"] = _normal((B, S, Hi), g, device)
        x["inorm_w"] = torch.ones(Di, device=device)
    x["sink"] = _normal((H,), g, device) if sink else None
    if wo_a:
        x["wo_a"] = _normal((O_GROUPS, (H // O_GROUPS) * D, O_RANK), g, device, 0.02).to(dt)
    else:
        x["wo_a"] = None
    return x


def make_entries(p, device="cpu", seed=3):
    """Stand-in for compressor output when the attention is tested alone:
    unit-RMS N(0,1) rows [B, S // ratio, D] in the storage dtype (the
    compressor's entries are RMS-normalised rows)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    N = p["S"] // p["ratio"] if p["ratio"] > 0 else 0
    return _unit_rms(_normal((p["B"], N, p["D"]), g, device)).to(torch_dtype(p))


def make_indexer_operands(p, device="cpu", seed=11):
    """Stand-in for the prepared indexer queries, the index keys and the head
    weights when the selection is tested alone: unit-RMS N(0,1) rows
    iq~ [B,S,Hi,Di] and ikey [B,S//ratio,Di] in the storage dtype, and
    w ~ N(0,1) [B,S,Hi] in float32, drawn in that order."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B, S, Hi, Di = p["B"], p["S"], p["Hi"], p["Di"]
    dt = torch_dtype(p)
    iqp = _unit_rms(_normal((B, S, Hi, Di), g, device)).to(dt)
    ikey = _unit_rms(_normal((B, S // p["ratio"], Di), g, device)).to(dt)
    w = _normal((B, S, Hi), g, device)
    return iqp, ikey, w


def make_output_grad(p, device="cpu", seed=2):
    """Gradient of the attention output for the backward: unit-RMS rows of
    N(0,1), [B,S,H,D] in the preset's storage dtype."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return _unit_rms(_normal((p["B"], p["S"], p["H"], p["D"]), g, device)).to(torch_dtype(p))


def random_topk_indices(B, S, ratio, K, device="cpu", seed=1):
    """Random valid selections: query t gets min(K, n_vis) distinct visible
    entries in random order, the rest of its row is -1 (random padding slots).

    Stands in for indexer output when the attention kernel is tested alone.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = torch.full((B, S, K), -1, dtype=torch.int32)
    for b in range(B):
        for t in range(S):
            nv = (t + 1) // ratio
            if nv == 0:
                continue
            take = min(K, nv)
            sel = torch.randperm(nv, generator=g)[:take].to(torch.int32)
            slots = torch.randperm(K, generator=g)[:take]
            out[b, t, slots] = sel
    return out.to(device)


def to_numpy64(t):
    """float64 numpy copy of a tensor (None passes through)."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()
