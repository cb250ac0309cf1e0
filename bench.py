#!/usr/bin/env python
"""Throughput of the DeepSeek-V4-Flash compressed attention forward on GB300.

One step = one CSA layer forward plus one HCA layer forward (the repeating
pair of the Flash stack), B=1, S=16384, 64 heads, 512-d latent, bf16, inputs
resident in HBM (q and o alone are 1 GiB each per layer, far above the 129 MB
L2, so no flush is needed).  value = tokens through the pair per second.
With N GPUs (``--gpus N``, one rank per GPU) the sequence's query rows are
split zig-zag across the ranks, balanced by per-row cost; every rank holds the
whole key/value prefix and computes only its rows (strong scaling, no
collective on the data path).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "attention-layer fwd tokens/s at S=16K (CSA & HCA)"
def workload(S):
    return ("DeepSeek-V4-Flash attention layer pair fwd: CSA (ratio 4 overlapped, indexer 64x128 "
            "fp32 scoring, top-512, window 128) + HCA (ratio 128, window 128), B=1, S=%d, "
            "H=64, D=512, R=64, bf16" % S)


# ---------------------------------------------------------------------------
# Algorithmic work (causal-exact) of one layer
# ---------------------------------------------------------------------------
def n_visible(t, r):
    return (t + 1) // r if r > 0 else 0


def attention_keys_total(S, r, K, W, lo=0, hi=None):
    """Keys read by the query positions lo..hi-1 (default all S)."""
    t = np.arange(lo, S if hi is None else hi, dtype=np.int64)
    nv = (t + 1) // r if r > 0 else np.zeros(len(t), dtype=np.int64)
    ne = np.minimum(nv, K) if K > 0 else nv
    nw = np.minimum(t + 1, W) if W >= 0 else t + 1
    return int((ne + nw).sum())


def layer_work(p, chunks=None):
    """Algorithmic work of one layer over the query positions in `chunks`
    (a list of [a, b) ranges; default the whole sequence).  A chunk's call
    reads the sequence side (kv, the compressors' inputs) up to its end."""
    B, S, H, D, r, K, W = p["B"], p["S"], p["H"], p["D"], p["ratio"], p["K"], p["W"]
    chunks = [(0, S)] if chunks is None else chunks
    keys = sum(attention_keys_total(S, r, K, W, a, b) for a, b in chunks)
    rows = sum(b - a for a, b in chunks)
    attn_flops = 4.0 * B * H * D * keys
    attn_bytes = 2.0 * B * rows * H * D * 2          # q read + o written (bf16)
    idx_pairs = 0
    if r > 0 and K > 0:
        idx_pairs = sum(int(((np.arange(a, b, dtype=np.int64) + 1) // r).sum()) for a, b in chunks)
    idx_flops = 2.0 * B * p["Hi"] * p["Di"] * idx_pairs
    # the layer's algorithmic HBM bytes: its inputs read once (q, kv, the
    # compressors' projections and scores, the indexer's queries and weights)
    # and its outputs written once (o, the selection)
    G = 1 + p["overlap"] if r > 0 else 0
    prefix = sum(b for _, b in chunks)               # sequence-side tokens read by the calls
    layer_bytes = attn_bytes + B * prefix * D * 2 + 2 * B * prefix * G * D * 2
    if r > 0 and K > 0:
        Hi, Di = p["Hi"], p["Di"]
        layer_bytes += B * rows * Hi * Di * 2 + 2 * B * prefix * G * Di * 2 + B * rows * Hi * 4 + B * rows * K * 4
    return dict(attn_flops=attn_flops, attn_bytes=attn_bytes, attn_keys=keys * B,
                idx_flops=idx_flops, idx_pairs=idx_pairs * B,
                layer_flops=attn_flops + idx_flops, layer_bytes=float(layer_bytes))


def layer_roofline(name, w, kernel_ms, peaks):
    """A whole layer against its roofline: the larger of its tensor time
    (FLOPs at the bf16 peak) and its HBM time (algorithmic bytes at the copy
    bandwidth), over the sum of the layer's kernel times."""
    t_tc = w["layer_flops"] / (peaks["bf16"] * 1e12) * 1e3
    t_hbm = w["layer_bytes"] / (peaks["hbm"] * 1e9) * 1e3
    return {"layer": name, "bound": "tensor" if t_tc >= t_hbm else "hbm", "ms": round(kernel_ms, 4),
            "bound_ms": round(max(t_tc, t_hbm), 4), "frac": round(max(t_tc, t_hbm) / kernel_ms, 4),
            "flops": w["layer_flops"], "bytes": w["layer_bytes"]}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# from an ncu capture of a smaller case of the same step: (kernel source, its
# sha256, bytes, sequence length of the capture).  The attention kernel's
# traffic is q + o, proportional to the query rows, so it is scaled by
# S / capture length.  A figure is reported only while its kernel source is
# unchanged.
NCU_TRAFFIC = {
    "csa_attention": ("mqa_tc.cu", "758f21ab174dce6f6663aa4a8742805787fdc833af4c7b4cc7fe5bd0bf72bc74",
                      507511296, 4096),
    "hca_attention": ("mqa_tc.cu", "758f21ab174dce6f6663aa4a8742805787fdc833af4c7b4cc7fe5bd0bf72bc74",
                      493794560, 4096),
}


TRAFFIC_SOURCE = ("dram__bytes_read.sum + dram__bytes_write.sum of one launch from an ncu capture of the same "
                  "kernel source on the B=1, S=4096 step, scaled by the query rows B*S / 4096 (the kernel's DRAM "
                  "traffic is q + o); a constant keyed to the source hash, not measured in this run; null when "
                  "the kernel changed since")


def traffic_fields(key, seq, world):
    """The roofline's traffic and where it comes from (null with the reason
    when no capture of the kernel's current source exists)."""
    t = ncu_traffic(key, seq) if world == 1 else None
    if t is not None:
        return {"traffic": t, "traffic_source": TRAFFIC_SOURCE}
    why = ("no DRAM capture of this kernel's current source" if world == 1 else
           "not given for a row slice (the capture covers whole-sequence launches)")
    return {"traffic": None, "traffic_source": why}


def ncu_traffic(key, seq):
    import hashlib
    if key not in NCU_TRAFFIC:
        return None
    src, sha, val, seq0 = NCU_TRAFFIC[key]
    path = os.path.join(ROOT, "sparse_compressed_attention_gb300", "csrc", src)
    try:
        cur = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    return int(round(val * seq / seq0)) if cur == sha else None


def indexer_unit(flops, scores_ms, topk_ms, peak):
    """The indexer as one unit: the score products' FLOPs over the time of
    the score kernel and the top-k selection that follows it."""
    ms = scores_ms + topk_ms
    tf = flops / (ms / 1e3) / 1e12
    return {"kernel": "csa indexer unit (scores + top-k)", "bound": "tensor", "achieved": round(tf, 2),
            "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(tf / peak, 4), "flops": flops,
            "scores_ms": round(scores_ms, 4), "topk_ms": round(topk_ms, 4)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d["bf16_tflops_sustained"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        self.file.flush()
        rows = []
        for line in open(self.file.name):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[6:10]))
            except Exception:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        use = inside if inside else sorted(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))[:3]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[3][i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_inside_timed_region": len(inside)}


# ---------------------------------------------------------------------------
# Distributed helpers (one process per GPU; timing protocol only)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def smi_index(local):
    """nvidia-smi index of this rank's GPU (honours CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in vis.split(",") if v.strip()]
    if local < len(ids):
        return ids[local]
    return str(local)


def max_over_ranks(value, device=None):
    """Max of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, device=None):
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def make_layer(name, S, device, seed, indexer_fp8=0, **over):
    import torch

    import seeded_inputs as SI
    import sparse_compressed_attention_gb300 as V
    p = SI.preset(name, S=S, **over)
    x = SI.make_layer_inputs(p, device, seed=seed)
    yarn = p["yarn"]
    f = V.v4_rope_inv_freq(p["theta"], p["R"], yarn, SI.YARN_ORIGINAL_LEN if yarn > 1 else 0,
                           SI.YARN_BETA_FAST, SI.YARN_BETA_SLOW).to(device)
    x["inv_freq"] = f
    cfg = V.config_from_preset(p, indexer_fp8=int(indexer_fp8) if p["K"] > 0 else 0)
    B, H = p["B"], p["H"]
    outs = {"o": torch.empty_like(x["q"]), "lse": torch.empty(B, S, H, device=device)}
    if p["K"] > 0:
        outs["idx"] = torch.empty(B, S, p["K"], dtype=torch.int32, device=device)
    ws = V.alloc_workspace(cfg, device)
    return dict(name=name, p=p, x=x, outs=outs, cfg=cfg, ws=ws)


def run_layer(L, stream=None):
    import sparse_compressed_attention_gb300 as V
    V.v4_attn_layer_fwd(L["cfg"], L["x"], L["outs"], L["ws"], stream)


ROW_INPUTS = ("q", "iq", "w")                           # one row per query position
SEQ_INPUTS = ("kv", "ckv", "cscore", "ickv", "icscore")  # one row per token of the sequence


def slice_layer(L, a, b):
    """The call of layer L over query positions [a, b): its own copies of
    the row inputs, the sequence inputs up to token b-1 (causality), its own
    outputs and workspace.  [0, S) is the layer itself."""
    import torch

    import sparse_compressed_attention_gb300 as V
    p = L["p"]
    if (a, b) == (0, p["S"]):
        return dict(L, chunk=(a, b))
    cfg = V.config_from_preset(p, S=b, q_begin=a, indexer_fp8=L["cfg"].indexer_fp8)
    x = {}
    for k, v in L["x"].items():
        if v is not None and k in ROW_INPUTS:
            x[k] = v[:, a:b].clone()             # own allocation: 16-byte aligned
        elif v is not None and k in SEQ_INPUTS:
            x[k] = v[:, :b].contiguous()
        else:
            x[k] = v
    B, H, dev = p["B"], p["H"], x["q"].device
    outs = {"o": torch.empty(B, b - a, H, p["D"], dtype=x["q"].dtype, device=dev),
            "lse": torch.empty(B, b - a, H, device=dev)}
    if p["K"] > 0:
        outs["idx"] = torch.empty(B, b - a, p["K"], dtype=torch.int32, device=dev)
    return dict(name=L["name"], p=p, x=x, outs=outs, cfg=cfg, ws=V.alloc_workspace(cfg, dev), chunk=(a, b))


def rank_chunks(p, world, rank, split="contiguous"):
    """This rank's query positions of one layer, balanced by the layer's
    per-row cost: one contiguous range, or the zig-zag pair of chunks (the
    whole sequence at N=1)."""
    from sparse_compressed_attention_gb300 import rows as R
    cost = R.layer_cost(p["ratio"], p["K"], p["W"], heads=p["H"], dim=p["D"], idx_heads=p["Hi"], idx_dim=p["Di"],
                        tile=128)
    if world == 1:
        return [(0, p["S"])]
    if split == "zigzag":
        return R.zigzag_chunks(p["S"], world, rank, cost)
    return R.contiguous_chunks(p["S"], world, rank, cost)


def relaunch_under_torchrun(args):
    """`--gpus N` without a launcher: start N ranks on this node (one per GPU)
    with torch.distributed.run and return its exit code."""
    import socket
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=%d" % args.gpus,
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import sparse_compressed_attention_gb300 as V
    from sparse_compressed_attention_gb300 import build as B
    ws_, rank, local = dist_env()
    if ws_ > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or local == 0:
        B.build()
    barrier()
    V.lib()
    S = args.seq
    # one sequence, the same inputs on every rank; each rank computes its
    # zig-zag share of the query rows of each layer against the whole prefix
    full = [make_layer("csa_bf16_16k", S, dev, seed=1000), make_layer("hca_bf16_16k", S, dev, seed=1001)]
    # --shard-of r/n (one process): time rank r's rows of an n-GPU split alone
    split_world, split_rank = ws_, rank
    if args.shard_of:
        split_rank, split_world = (int(v) for v in args.shard_of.split("/"))
        if ws_ > 1 or not 0 <= split_rank < split_world:
            raise SystemExit("--shard-of r/n needs one process and 0 <= r < n")
    chunks_of = {L["name"]: rank_chunks(L["p"], split_world, split_rank, args.split) for L in full}
    layers = [slice_layer(L, a, b) for L in full for a, b in chunks_of[L["name"]]]
    if split_world > 1:
        for L in full:                       # the whole-sequence outputs are not used by a rank
            L["outs"] = None
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        for L in layers:
            run_layer(L)
    torch.cuda.synchronize(dev)

    clk = ClockSampler(smi_index(local))
    clk.start()
    # keep the GPU busy briefly so the sampler sees load before the timed region
    t_pre = time.time()
    while time.time() - t_pre < 0.3:
        for L in layers:
            run_layer(L)
        torch.cuda.synchronize(dev)
    # the step as one CUDA graph: the library's calls are captured once (no
    # host work per step), each replay launches the same kernels
    graph, graph_note, per_step = None, None, 0
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            l0 = V.v4_launch_count()
            with torch.cuda.graph(g):
                for L in layers:
                    run_layer(L)
            per_step = V.v4_launch_count() - l0
            g.replay()
            torch.cuda.synchronize(dev)
            graph = g
        except Exception as exc:             # capture refused: time the eager calls
            graph_note = "graph capture failed: %s" % str(exc).splitlines()[0][:120]
    marks = []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph is None:
        V.v4_profile_enable(True)
    launches0 = V.v4_launch_count()
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
            continue
        for L in layers:
            run_layer(L)
            marks.append((L["name"], V.v4_profile_count()))
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier()
    launches = per_step * args.steps if graph is not None else V.v4_launch_count() - launches0
    if graph is not None:
        # per-kernel durations from an eager pass with the library's events
        V.v4_profile_enable(True)
        for _ in range(args.steps):
            for L in layers:
                run_layer(L)
                marks.append((L["name"], V.v4_profile_count()))
        torch.cuda.synchronize(dev)
    V.v4_profile_enable(False)
    clk.stop()
    clocks = clk.summary(t0, t1)
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, dev)
    status = V.v4_get_device_status()

    # per-kernel durations from the live event records (of the timed region
    # itself when the step runs eagerly); a kernel's time per step sums its
    # launches over this rank's row chunks of the layer
    recs = V.v4_profile_records()
    per = {}
    start = 0
    for name, end in marks:
        for kind, t in recs[start:end]:
            per.setdefault((name, kind), []).append(t)
        start = end
    kern = {"%s/%s" % k: {"launches": len(v), "avg_ms": sum(v) / len(v), "total_ms": sum(v)}
            for k, v in per.items()}

    def per_step_ms(key):
        v = per.get(key, [])
        return sum(v) / args.steps if v else None

    # tokens through the layer pair: this rank's rows (each layer's chunks
    # cover the sequence once over all ranks)
    rows = {n: sum(b - a for a, b in ch) for n, ch in chunks_of.items()}
    tokens_rank = full[0]["p"]["B"] * (rows["csa_bf16_16k"] + rows["hca_bf16_16k"]) / 2.0
    tokens = sum_over_ranks(tokens_rank * args.steps, dev)
    value = tokens / (ms / 1e3)

    peaks = load_peaks()
    work = {L["name"]: layer_work(L["p"], chunks_of[L["name"]]) for L in full}
    nlaunch = {n: len(ch) for n, ch in chunks_of.items()}
    roof = None
    a_ms = per_step_ms(("csa_bf16_16k", "attention"))
    if a_ms:
        achieved = work["csa_bf16_16k"]["attn_flops"] / (a_ms / 1e3) / 1e12
        roof = {"kernel": "csa attention (sparse MQA, 64 heads x 512, top-512 + window 128)",
                "bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16"], 4),
                **traffic_fields("csa_attention", S, ws_),
                "peak_source": "%s bf16 burst (MEASURED_PEAKS.json)" % peaks["src"],
                "flops_per_launch": work["csa_bf16_16k"]["attn_flops"] / nlaunch["csa_bf16_16k"],
                "avg_launch_ms": round(a_ms / nlaunch["csa_bf16_16k"], 4),
                "launches_per_step": nlaunch["csa_bf16_16k"]}
    extra_roofs = []
    a_ms = per_step_ms(("hca_bf16_16k", "attention"))
    if a_ms:
        gbs = work["hca_bf16_16k"]["attn_bytes"] / (a_ms / 1e3) / 1e9
        extra_roofs.append({"kernel": "hca attention", "bound": "hbm", "achieved": round(gbs, 1),
                            "peak": peaks["hbm"], "unit": "GB/s", "frac": round(gbs / peaks["hbm"], 4),
                            **traffic_fields("hca_attention", S, ws_),
                            "bytes_per_launch": work["hca_bf16_16k"]["attn_bytes"] / nlaunch["hca_bf16_16k"],
                            "avg_launch_ms": round(a_ms / nlaunch["hca_bf16_16k"], 4),
                            "launches_per_step": nlaunch["hca_bf16_16k"]})
    s_ms = per_step_ms(("csa_bf16_16k", "indexer_scores"))
    if s_ms:
        tf = work["csa_bf16_16k"]["idx_flops"] / (s_ms / 1e3) / 1e12
        extra_roofs.append({"kernel": "csa indexer scores", "bound": "tensor", "achieved": round(tf, 2),
                            "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": round(tf / peaks["bf16"], 4),
                            **traffic_fields("csa_indexer", S, ws_),
                            "flops_per_launch": work["csa_bf16_16k"]["idx_flops"] / nlaunch["csa_bf16_16k"],
                            "avg_launch_ms": round(s_ms / nlaunch["csa_bf16_16k"], 4)})
        tk = per_step_ms(("csa_bf16_16k", "topk"))
        if tk:
            extra_roofs.append(indexer_unit(work["csa_bf16_16k"]["idx_flops"], s_ms, tk, peaks["bf16"]))
            pr = per_step_ms(("csa_bf16_16k", "indexer_prep"))
            if pr:
                u = indexer_unit(work["csa_bf16_16k"]["idx_flops"], s_ms + pr, tk, peaks["bf16"])
                u["kernel"] = "csa indexer unit with its query prep (prep + scores + top-k)"
                u["prep_ms"] = round(pr, 4)
                u["scores_ms"] = round(s_ms, 4)
                extra_roofs.append(u)

    layer_roofs = []
    for name in work:
        tot = sum(sum(v) for (n, k), v in per.items() if n == name)      # every launch of the profiled steps
        if tot > 0:
            layer_roofs.append(layer_roofline(name, work[name], tot / args.steps, peaks))

    e2e = run_e2e(args, layers, dev, tokens_rank) if args.e2e_steps > 0 else None

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws_,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; activations unit-RMS N(0,1), q from a random rank-1024 path)",
        "config": {"workload": workload(S), "global_batch": 1, "seq_len": S, "layers_per_step": 2,
                   "cuda_graph": graph is not None,
                   "parallelism": ("query rows of one sequence split over %d GPUs (%s, cost-balanced), "
                                   "no collective on the data path" % (ws_, args.split)) if ws_ > 1 else "single",
                   "rank0_chunks": {n: [list(c) for c in ch] for n, ch in chunks_of.items()},
                   "shard_of": args.shard_of or None,
                   "l2": "no flush: inputs larger than L2 (q and o 1 GiB per layer)"},
        "clocks": clocks, "gpu_launches": launches, "device_status": status,
        "roofline": roof, "roofline_other": extra_roofs, "roofline_layers": layer_roofs, "kernels": kern,
        "e2e": e2e,
    }
    if graph_note:
        line["note"] = graph_note
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, full)
    if ws_ == 1 and not args.shard_of and args.configs:
        # the benchmark's other configurations, after the headline timing
        del layers, full
        torch.cuda.empty_cache()
        line["configs"] = {k: measure_config(k, dev, args, peaks) for k in args.configs.split(",") if k}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_ > 1:
        dist.destroy_process_group()


def run_e2e(args, layers, dev, tokens_rank):
    """Same step through the C ABI with inputs in pinned host memory: every
    step copies every input of both layers host->device and each layer's
    output o device->host.  Copies in and out run on their own streams and
    overlap the other layer's compute: a layer's inputs are refilled once its
    previous compute is done with them, and its o buffer is rewritten only
    after the previous read-back has finished."""
    import torch
    hosts = []
    h2d = d2h = 0
    for L in layers:
        hx = {k: (v.to("cpu").pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in L["x"].items()}
        ho = L["outs"]["o"].to("cpu").pin_memory()
        hosts.append((hx, ho))
        h2d += sum(v.numel() * v.element_size() for v in hx.values() if isinstance(v, torch.Tensor))
        d2h += ho.numel() * ho.element_size()
    n = args.e2e_steps
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done = [None] * len(layers)       # compute of layer i finished (inputs free)
    read = [None] * len(layers)       # read-back of layer i's o finished (o free)

    def step():
        for i, (L, (hx, ho)) in enumerate(zip(layers, hosts)):
            with torch.cuda.stream(s_in):
                if done[i] is not None:
                    s_in.wait_event(done[i])
                for k, v in hx.items():
                    if isinstance(v, torch.Tensor):
                        L["x"][k].copy_(v, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            comp.wait_event(ready)
            if read[i] is not None:
                comp.wait_event(read[i])
            run_layer(L, comp.cuda_stream)
            done[i] = torch.cuda.Event()
            done[i].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[i])
                ho.copy_(L["outs"]["o"], non_blocking=True)
                read[i] = torch.cuda.Event()
                read[i].record(s_out)

    # one untimed pass through the same pipeline (first use of the pinned
    # buffers), then n timed steps starting from an empty pipeline
    step()
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    torch.cuda.synchronize(dev)
    done = [None] * len(layers)
    read = [None] * len(layers)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    for _ in range(n):
        step()
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    e1.record(comp)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    tokens = sum_over_ranks(tokens_rank * n, dev)
    return {"value": round(tokens / (ms / 1e3), 1), "unit": "tokens/s", "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "copies in and out on their own streams, overlapping the other layer's compute"}


# ---------------------------------------------------------------------------
# Other workloads (not the default line): the 43-layer Flash stack with the
# grouped output projection, and a single CSA layer (the long-context case)
# ---------------------------------------------------------------------------
STACK_ORDER = ["swa", "swa"] + ["csa", "hca"] * 20 + ["csa"]      # 2 SWA + 21 CSA + 20 HCA


def make_stack_layer(kind, B, S, device, seed):
    import torch

    import seeded_inputs as SI
    import sparse_compressed_attention_gb300 as V
    name = {"swa": "swa_bf16_16k", "csa": "csa_bf16_16k", "hca": "hca_bf16_16k"}[kind]
    p = SI.preset(name, B=B, S=S)
    x = SI.make_layer_inputs(p, device, seed=seed, wo_a=True)
    yarn = p["yarn"]
    x["inv_freq"] = V.v4_rope_inv_freq(p["theta"], p["R"], yarn, SI.YARN_ORIGINAL_LEN if yarn > 1 else 0,
                                       SI.YARN_BETA_FAST, SI.YARN_BETA_SLOW).to(device)
    cfg = V.config_from_preset(p)
    H = p["H"]
    outs = {"o": torch.empty_like(x["q"]), "lse": torch.empty(B, S, H, device=device),
            "y": torch.empty(B, S, x["wo_a"].shape[0] * x["wo_a"].shape[2], dtype=x["q"].dtype, device=device)}
    if p["K"] > 0:
        outs["idx"] = torch.empty(B, S, p["K"], dtype=torch.int32, device=device)
    return dict(name=kind, p=p, x=x, outs=outs, cfg=cfg, ws=V.alloc_workspace(cfg, device))


def run_qproj(args):
    """--workload qproj: the query projections of the rank-1024 latent (q with
    per-head RMSNorm, and the indexer queries) for B=1, S tokens."""
    import torch

    import seeded_inputs as SI
    import sparse_compressed_attention_gb300 as V
    from sparse_compressed_attention_gb300 import build as Bld
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    Bld.build()
    V.lib()
    S = args.seq
    p = SI.preset("csa_bf16_16k", S=S)
    H, D, Hi, Di, rank = p["H"], p["D"], p["Hi"], p["Di"], SI.Q_RANK
    g = torch.Generator(device=dev).manual_seed(5000)
    qlat = torch.randn(1, S, rank, generator=g, device=dev).to(torch.bfloat16)
    wq = (torch.randn(rank, H * D, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    wiq = (torch.randn(rank, Hi * Di, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    q = torch.empty(1, S, H, D, dtype=torch.bfloat16, device=dev)
    iq = torch.empty(1, S, Hi, Di, dtype=torch.bfloat16, device=dev)
    cfg = V.config_from_preset(p)
    for _ in range(args.warmup):
        V.v4_q_proj(cfg, qlat, wq, q, 1, None, wiq, iq)
    torch.cuda.synchronize(dev)
    clk = ClockSampler(smi_index(0))
    clk.start()
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = V.v4_launch_count()
    t0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        V.v4_q_proj(cfg, qlat, wq, q, 1, None, wiq, iq)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    clk.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    flops = 2.0 * S * rank * (H * D + Hi * Di)
    tf = flops / (ms / 1e3) / 1e12
    peaks = load_peaks()
    line = {"metric": "query projection tokens/s at S=%d (rank-1024 latent -> 64x512 q, 64x128 iq)" % S,
            "value": round(S / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) latent, N(0,0.02) weights)",
            "config": {"workload": "q and indexer-q projections of the rank-1024 latent, per-head RMSNorm on q, "
                                   "B=1, S=%d" % S, "global_batch": 1, "seq_len": S},
            "clocks": clk.summary(t0, t1), "gpu_launches": V.v4_launch_count() - launches0,
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                         "frac": round(tf / peaks["bf16"], 4), "traffic": None,
                         "traffic_source": "no DRAM capture of this kernel's current source",
                         "flops_per_launch": flops}}
    print(json.dumps(line), flush=True)


def run_kl(args):
    """--workload kl: the sparse indexer distillation target (target, KL loss
    and its gradient) of the CSA layer at B=1, S tokens, after one forward of
    the layer has produced the selections, their scores, the entries and lse."""
    import torch

    import sparse_compressed_attention_gb300 as V
    from sparse_compressed_attention_gb300 import build as Bld
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    Bld.build()
    V.lib()
    S = args.seq
    L = make_layer("csa_bf16_16k", S, dev, seed=6000)
    p, x, outs = L["p"], L["x"], L["outs"]
    B, H, K = p["B"], p["H"], p["K"]
    outs["ent"] = torch.empty(B, S // p["ratio"], p["D"], dtype=torch.bfloat16, device=dev)
    outs["iscore"] = torch.empty(B, S, K, device=dev)
    run_layer(L)
    target = torch.empty(B, S, K, device=dev)
    loss = torch.empty(B, S, device=dev)
    dscore = torch.empty(B, S, K, device=dev)
    args_ = (L["cfg"], x["q"], outs["ent"], outs["idx"], outs["lse"], outs["iscore"], x["inv_freq"], target, loss,
             dscore, L["ws"])
    for _ in range(args.warmup):
        V.v4_indexer_kl_target(*args_)
    torch.cuda.synchronize(dev)
    clk = ClockSampler(smi_index(0))
    clk.start()
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = V.v4_launch_count()
    t0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        V.v4_indexer_kl_target(*args_)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    clk.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    pairs = int((outs["idx"] >= 0).sum().item())
    flops = 2.0 * H * p["D"] * pairs                 # the logits of every (query, selected entry)
    tf = flops / (ms / 1e3) / 1e12
    peaks = load_peaks()
    line = {"metric": "indexer distillation target tokens/s at S=%d (CSA, top-%d)" % (S, K),
            "value": round(B * S / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; the layer's own selections)",
            "config": {"workload": "sparse indexer KL target, loss and gradient of one CSA layer, B=1, S=%d, "
                                   "H=64, D=512, top-%d" % (S, K), "global_batch": B, "seq_len": S,
                       "selected_pairs": pairs},
            "clocks": clk.summary(t0, t1), "gpu_launches": V.v4_launch_count() - launches0,
            "device_status": V.v4_get_device_status(),
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                         "frac": round(tf / peaks["bf16"], 4), "traffic": None,
                         "traffic_source": "no DRAM capture of this kernel's current source",
                         "flops_per_launch": flops}}
    print(json.dumps(line), flush=True)


def run_workload(args):
    """--workload stack | csa: one JSON line for that workload (1 GPU)."""
    import torch

    import sparse_compressed_attention_gb300 as V
    from sparse_compressed_attention_gb300 import build as Bld
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    Bld.build()
    V.lib()
    S = args.seq
    if args.workload == "pro":
        B = 1
        order = [make_layer("csa_bf16_16k", S, dev, seed=4000, H=128, K=1024),
                 make_layer("hca_bf16_16k", S, dev, seed=4001, H=128)]
        order[0]["name"], order[1]["name"] = "csa", "hca"
        metric = "attention-layer fwd tokens/s at S=%d (CSA & HCA), 128 heads, top-1024" % S
        wl = ("DeepSeek-V4-Pro-like attention layer pair fwd (128 heads, top-1024; other shapes as Flash), "
              "B=1, S=%d, H=128, D=512, R=64, bf16" % S)
    elif args.workload == "stack":
        B = 2
        kinds = {k: make_stack_layer(k, B, S, dev, seed=2000 + i) for i, k in enumerate(("swa", "csa", "hca"))}
        order = [kinds[k] for k in STACK_ORDER]
        metric = "Flash stack fwd tokens/s (43 layers: 2 SWA + 21 CSA + 20 HCA, grouped wo_a)"
        wl = ("DeepSeek-V4-Flash 43-layer attention stack fwd with the 8-group x 1024 grouped O projection, "
              "B=%d, S=%d, H=64, D=512, R=64, bf16" % (B, S))
    else:
        B = 1
        order = [make_layer("csa_bf16_16k", S, dev, seed=3000, indexer_fp8=args.indexer_fp8)]
        for L in order:
            L["name"] = "csa"
        metric = "CSA layer fwd tokens/s at S=%d" % S
        scoring = "E4M3 operands, per-row scales" if args.indexer_fp8 else "bf16 operands"
        wl = ("DeepSeek-V4-Flash CSA layer fwd (ratio 4 overlapped, indexer 64x128 %s, fp32 scoring, top-512, "
              "window 128), B=1, S=%d, H=64, D=512, R=64, bf16" % (scoring, S))
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        for L in order:
            run_layer(L)
    torch.cuda.synchronize(dev)
    clk = ClockSampler(smi_index(0))
    clk.start()
    t_pre = time.time()
    while time.time() - t_pre < 0.3:
        for L in order:
            run_layer(L)
        torch.cuda.synchronize(dev)
    V.v4_profile_enable(True)
    launches0 = V.v4_launch_count()
    marks = []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        for L in order:
            run_layer(L)
            marks.append((L["name"], V.v4_profile_count()))
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    launches = V.v4_launch_count() - launches0
    V.v4_profile_enable(False)
    clk.stop()
    ms = ev0.elapsed_time(ev1)
    recs = V.v4_profile_records()
    per, start = {}, 0
    for name, end in marks:
        for kind, t in recs[start:end]:
            per.setdefault((name, kind), []).append(t)
        start = end
    kern = {"%s/%s" % k: {"launches": len(v), "avg_ms": sum(v) / len(v), "total_ms": sum(v)}
            for k, v in per.items()}
    peaks = load_peaks()
    csa = next(L for L in order if L["name"] == "csa")
    wk = layer_work(csa["p"])
    roof, other = None, []
    a = per.get(("csa", "attention"), [])
    if a:
        a_ms = sum(a) / len(a)
        tf = wk["attn_flops"] / (a_ms / 1e3) / 1e12
        roof = {"kernel": "csa attention", "bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16"],
                "unit": "TFLOP/s", "frac": round(tf / peaks["bf16"], 4),
                **traffic_fields("csa_attention", csa["p"]["B"] * csa["p"]["S"], 1),
                "flops_per_launch": wk["attn_flops"], "avg_launch_ms": round(a_ms, 4)}
    isc = per.get(("csa", "indexer_scores"), [])
    if isc:
        a_ms = sum(isc) / len(isc)
        tf = wk["idx_flops"] / (a_ms / 1e3) / 1e12
        fp8 = bool(csa["cfg"].indexer_fp8)
        # E4M3 products: the measured bf16 peak times the nominal e4m3/bf16 ratio (4.5 / 2.25)
        pk = peaks["bf16"] * (2.0 if fp8 else 1.0)
        other.append({"kernel": "csa indexer scores" + (" (E4M3)" if fp8 else ""), "bound": "tensor",
                      "achieved": round(tf, 2), "peak": round(pk, 1), "unit": "TFLOP/s",
                      "frac": round(tf / pk, 4), "flops_per_launch": wk["idx_flops"],
                      "avg_launch_ms": round(a_ms, 4)})
        tk = per.get(("csa", "topk"), [])
        if tk:
            other.append(indexer_unit(wk["idx_flops"], a_ms, sum(tk) / len(tk), pk))
    op = [t for (n, k), v in per.items() if k == "o_proj" for t in v]
    if op:
        a_ms = sum(op) / len(op)
        fl = 2.0 * B * S * 8 * 4096 * 1024
        tf = fl / (a_ms / 1e3) / 1e12
        other.append({"kernel": "grouped wo_a projection", "bound": "tensor", "achieved": round(tf, 2),
                      "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": round(tf / peaks["bf16"], 4),
                      "flops_per_launch": fl, "avg_launch_ms": round(a_ms, 4)})
    line = {"metric": metric, "value": round(B * S * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; activations unit-RMS N(0,1), q from a random rank-1024 path)",
            "config": {"workload": wl, "global_batch": B, "seq_len": S, "layers_per_step": len(order)},
            "clocks": clk.summary(t0, t1), "gpu_launches": launches,
            "device_status": V.v4_get_device_status(), "roofline": roof, "roofline_other": other,
            "kernels": kern}
    print(json.dumps(line), flush=True)



# ---------------------------------------------------------------------------
# The other workloads of the benchmark definition, measured in the same run
# (one GPU): the CSA layer at S=4096 and at S=65536, and the 43-layer stack at
# B=2 with the grouped output projection.  Each gets its tokens/s, its
# roofline and the oracle's time on a bounded sample.
# ---------------------------------------------------------------------------
EXTRA_CONFIGS = {
    "csa_s4096": dict(kind="csa", B=1, S=4096,
                      workload="DeepSeek-V4-Flash CSA layer fwd (ratio 4 overlapped, indexer 64x128 fp32 scoring, "
                               "top-512, window 128), B=1, S=4096, H=64, D=512, R=64, bf16"),
    "csa_s65536": dict(kind="csa", B=1, S=65536,
                       workload="DeepSeek-V4-Flash long-context CSA layer fwd (ratio 4 overlapped, indexer 64x128 "
                                "fp32 scoring, top-512, window 128), B=1, S=65536, H=64, D=512, R=64, bf16"),
    "stack_b2_s16384": dict(kind="stack", B=2, S=16384,
                            workload="DeepSeek-V4-Flash 43-layer attention stack fwd (2 SWA + 21 CSA + 20 HCA) with "
                                     "the 8-group x 1024 grouped O projection, B=2, S=16384, H=64, D=512, R=64, "
                                     "bf16"),
}
STACK_COUNTS = {"swa": 2, "csa": 21, "hca": 20}


def measure_config(key, dev, args, peaks):
    """Time one extra workload: warm-up, --cfg-steps timed steps (CUDA events
    on the launching stream), then one step with per-stage events."""
    import torch

    import sparse_compressed_attention_gb300 as V
    c = EXTRA_CONFIGS[key]
    B, S = c["B"], c["S"]
    if c["kind"] == "stack":
        kinds = {k: make_stack_layer(k, B, S, dev, seed=2000 + i) for i, k in enumerate(("swa", "csa", "hca"))}
        order = [kinds[k] for k in STACK_ORDER]
        counts = STACK_COUNTS
    else:
        L = make_layer("csa_bf16_16k", S, dev, seed=3000)
        L["name"] = "csa"
        kinds, order, counts = {"csa": L}, [L], {"csa": 1}
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.cfg_warmup):
        for L in order:
            run_layer(L)
    torch.cuda.synchronize(dev)
    clk = ClockSampler(smi_index(dev.index or 0))
    clk.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    ev0.record(stream)
    for _ in range(args.cfg_steps):
        for L in order:
            run_layer(L)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    clk.stop()
    ms = ev0.elapsed_time(ev1) / args.cfg_steps
    V.v4_profile_enable(True)
    marks = []
    for L in order:
        run_layer(L)
        marks.append((L["name"], V.v4_profile_count()))
    torch.cuda.synchronize(dev)
    recs = V.v4_profile_records()
    V.v4_profile_enable(False)
    per, start = {}, 0
    for name, end in marks:
        for kind, t in recs[start:end]:
            per.setdefault((name, kind), []).append(t)
        start = end
    entry = {"workload": c["workload"], "value": round(B * S / (ms / 1e3), 1), "unit": "tokens/s",
             "ms_per_step": round(ms, 4), "steps": args.cfg_steps, "warmup": args.cfg_warmup,
             "global_batch": B, "seq_len": S, "layers_per_step": len(order), "clocks": clk.summary(t0, t1)}
    wk = layer_work(kinds["csa"]["p"])
    a = per.get(("csa", "attention"), [])
    if a:
        a_ms = sum(a) / len(a)
        tf = wk["attn_flops"] / (a_ms / 1e3) / 1e12
        entry["roofline"] = {"kernel": "csa attention", "bound": "tensor", "achieved": round(tf, 2),
                             "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": round(tf / peaks["bf16"], 4),
                             "flops_per_launch": wk["attn_flops"], "avg_launch_ms": round(a_ms, 4),
                             **traffic_fields("csa_attention", B * S, 1)}
    isc, tk = per.get(("csa", "indexer_scores"), []), per.get(("csa", "topk"), [])
    if isc and tk:
        entry["roofline_indexer_unit"] = indexer_unit(wk["idx_flops"], sum(isc) / len(isc), sum(tk) / len(tk),
                                                      peaks["bf16"])
    if c["kind"] == "stack":
        # the whole stack against its roofline: every layer's FLOPs and bytes,
        # plus the projection's (2*B*S*8*4096*1024 FLOPs, its weights and y)
        fl = by = 0.0
        for k, n in counts.items():
            w = layer_work(kinds[k]["p"])
            fl += n * (w["layer_flops"] + 2.0 * B * S * 8 * 4096 * 1024)
            by += n * (w["layer_bytes"] + 8 * 4096 * 1024 * 2 + B * S * 8 * 1024 * 2)
        t_tc, t_hbm = fl / (peaks["bf16_sustained"] * 1e12) * 1e3, by / (peaks["hbm"] * 1e9) * 1e3
        entry["roofline_stack"] = {"bound": "tensor" if t_tc >= t_hbm else "hbm", "flops": fl, "bytes": by,
                                   "bound_ms": round(max(t_tc, t_hbm), 4), "ms": round(ms, 4),
                                   "frac": round(max(t_tc, t_hbm) / ms, 4),
                                   "peak_source": "bf16 sustained (a long step) and HBM copy, MEASURED_PEAKS.json"}
        op = [t for (n, k), v in per.items() if k == "o_proj" for t in v]
        if op:
            o_ms = sum(op) / len(op)
            fl1 = 2.0 * B * S * 8 * 4096 * 1024
            entry["roofline_o_proj"] = {"kernel": "grouped wo_a projection", "bound": "tensor",
                                        "achieved": round(fl1 / (o_ms / 1e3) / 1e12, 2), "peak": peaks["bf16"],
                                        "unit": "TFLOP/s",
                                        "frac": round(fl1 / (o_ms / 1e3) / 1e12 / peaks["bf16"], 4),
                                        "avg_launch_ms": round(o_ms, 4)}
    if not args.no_cpu_baseline:
        rows = 16
        while True:
            inputs = gather_oracle_inputs(list(kinds.values()), rows)
            est, spent = oracle_sample(inputs, rows, counts)
            if spent >= args.cfg_cpu_seconds or rows >= S:
                break
            rows = min(S, rows * 2)
        entry["cpu_baseline"] = {"value": round(B * S / est, 3), "unit": "tokens/s", "cores": os.cpu_count(),
                                 "kind": "oracle",
                                 "sample": "numpy float64 oracle: full compressors + indexer/attention%s for %d evenly "
                                           "spaced query rows per layer kind, extrapolated to B=%d, S=%d%s (%.1f s of "
                                           "CPU work)" % (" + grouped projection" if c["kind"] == "stack" else "",
                                                          rows, B, S, " and the 2+21+20 layer mix"
                                                          if c["kind"] == "stack" else "", spent)}
    del order, kinds
    torch.cuda.empty_cache()
    return entry


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (rank 0 only)
# ---------------------------------------------------------------------------
def oracle_sample(inputs_by_layer, rows_per_layer, counts=None):
    """Time the oracle on: the full compressors of every layer, plus indexer,
    attention (and, with wo_a, the grouped projection) for `rows_per_layer`
    evenly spaced query rows per layer.  `counts` (name -> layers of that
    kind) scales each layer's estimate.  Returns (seconds extrapolated to all
    S rows of every layer, seconds spent)."""
    from oracle import v4_oracle as O
    total_est = 0.0
    spent = 0.0
    for name, (p, x) in inputs_by_layer.items():
        S = p["S"]
        rows = np.linspace(0, S - 1, rows_per_layer).round().astype(np.int64)
        ta = time.perf_counter()
        ent = ikey = None
        if p["ratio"] > 0:
            ent = O.compress(x["ckv"], x["cscore"], x["ape"], x["norm_w"], x["inv_freq"], p["ratio"],
                             p["overlap"], 1e-6, store_bf16=True)
        if p["K"] > 0:
            ikey = O.compress(x["ickv"], x["icscore"], x["iape"], x["inorm_w"], x["inv_freq"],
                              p["ratio"], p["overlap"], 1e-6, hadamard=True, store_bf16=True)
        tb = time.perf_counter()
        idx_rows = None
        if p["K"] > 0:
            sel = O.indexer_topk(x["iq_rows"], ikey, x["w_rows"], x["inv_freq"], p["ratio"], p["K"],
                                 store_bf16=True, rows=rows, rows_only=True)
            idx_rows = sel["idx"]
        o, _ = O.sparse_mqa(x["q_rows"], x["kv"], ent, idx_rows, None, x["inv_freq"], p["ratio"], p["W"],
                            store_bf16=True, rows=rows, rows_only=True)
        if x.get("wo_a") is not None:
            O.grouped_wo_a(o, x["wo_a"], store_bf16=True)
        tc = time.perf_counter()
        n = (counts or {}).get(name, 1)
        total_est += n * ((tb - ta) + (tc - tb) * S / len(rows))
        spent += tc - ta
    return total_est, spent


def gather_oracle_inputs(layers, rows_per_layer):
    import torch
    out = {}
    for L in layers:
        p, x = L["p"], L["x"]
        S = p["S"]
        rows = torch.from_numpy(np.linspace(0, S - 1, rows_per_layer).round().astype(np.int64))
        d = {k: x[k].detach().double().cpu().numpy() for k in
             ("kv", "ckv", "cscore", "ape", "norm_w", "wo_a") if x.get(k) is not None}
        d["inv_freq"] = x["inv_freq"].cpu().numpy()
        d["q_rows"] = x["q"][:, rows.to(x["q"].device)].double().cpu().numpy()
        if p["K"] > 0:
            for k in ("ickv", "icscore", "iape", "inorm_w"):
                d[k] = x[k].detach().double().cpu().numpy()
            d["iq_rows"] = x["iq"][:, rows.to(x["iq"].device)].double().cpu().numpy()
            d["w_rows"] = x["w"][:, rows.to(x["w"].device)].double().cpu().numpy()
        out[L["name"]] = (p, d)
    return out


def cpu_baseline(args, layers):
    """Oracle time on a sample sized to roughly 10-30 s of CPU work: the row
    count doubles until one sample takes at least --cpu-seconds."""
    S = layers[0]["p"]["S"]
    rows = args.cpu_rows
    while True:
        inputs = gather_oracle_inputs(layers, rows)
        est, spent = oracle_sample(inputs, rows)
        if spent >= args.cpu_seconds or rows >= S:
            break
        rows = min(S, rows * 2)
    return {"value": round(S / est, 2), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": "numpy float64 oracle: full compressors of both layers + indexer/attention for "
                      "%d evenly spaced query rows per layer, extrapolated to S=%d (%.1f s of CPU work)"
                      % (rows, S, spent)}


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle as the comparison program
# ---------------------------------------------------------------------------
def run_reference(args):
    """The CPU oracle as the comparison program, on the same workload.  One
    step = the oracle on a bounded sample (the full compressors of both layers
    and the indexer and attention of --ref-rows evenly spaced query rows per
    layer, as cpu_baseline samples them); ms_per_step is the measured time of
    that sample, value the whole-sequence throughput extrapolated from it."""
    import torch

    import seeded_inputs as SI
    from oracle import v4_oracle as O
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    S = args.seq
    layers = []
    for name, seed in (("csa_bf16_16k", 1000), ("hca_bf16_16k", 1001)):
        p = SI.preset(name, S=S)
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        x = SI.make_layer_inputs(p, dev, seed=seed)
        x["inv_freq"] = torch.from_numpy(O.make_inv_freq(p["theta"], p["R"], p["yarn"],
                                                         SI.YARN_ORIGINAL_LEN if p["yarn"] > 1 else 0))
        layers.append(dict(name=name, p=p, x=x))
    inputs = gather_oracle_inputs(layers, args.ref_rows)
    for _ in range(args.warmup):
        oracle_sample(inputs, args.ref_rows)
    ests, spent = [], []
    for _ in range(args.steps):
        e, sp = oracle_sample(inputs, args.ref_rows)
        ests.append(e)
        spent.append(sp)
    est = sum(ests) / len(ests)
    value = S / est
    sample = ("numpy float64 oracle per step: full compressors of both layers + indexer/attention for %d evenly "
              "spaced query rows per layer (the rows cpu_baseline samples), extrapolated to S=%d"
              % (args.ref_rows, S))
    cb = {"value": round(value, 2), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
          "sample": sample}
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * sum(spent) / len(spent), 1), "extrapolated": True,
            "extrapolated_ms_per_step": round(est * 1e3, 1), "sample_rows_per_layer": args.ref_rows,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload(S), "global_batch": 1, "seq_len": S, "layers_per_step": 2},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seq", type=int, default=16384)
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-rows", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager calls instead of a captured step")
    ap.add_argument("--configs", default="csa_s4096,csa_s65536,stack_b2_s16384",
                    help="extra workloads measured after the headline pair (one GPU), comma-separated; '' = none")
    ap.add_argument("--cfg-steps", type=int, default=5)
    ap.add_argument("--cfg-warmup", type=int, default=3)
    ap.add_argument("--cfg-cpu-seconds", type=float, default=4.0)
    ap.add_argument("--split", choices=["contiguous", "zigzag"], default="contiguous",
                    help="N > 1: how the query rows of the sequence are split (both balanced by per-row cost)")
    ap.add_argument("--shard-of", default="", help="r/n: one process times rank r's query rows of an n-GPU "
                                                   "split (value then counts only those rows)")
    ap.add_argument("--indexer-fp8", type=int, choices=[0, 1], default=0,
                    help="--workload csa: opt-in E4M3 indexer QK (the default keeps bf16 operands)")
    ap.add_argument("--workload", choices=["pair", "stack", "csa", "pro", "qproj", "kl"], default="pair",
                    help="pair: the CSA + HCA layer pair (the reported line); stack: the 43-layer "
                         "Flash stack with grouped wo_a at B=2; csa: one CSA layer (e.g. --seq 65536); "
                         "pro: the pair with 128 heads and top-1024; qproj: the rank-1024 query projections; "
                         "kl: the indexer distillation target of the CSA layer")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and args.impl == "ours" and args.workload == "pair":
        sys.exit(relaunch_under_torchrun(args))
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "qproj":
        run_qproj(args)
    elif args.workload == "kl":
        run_kl(args)
    elif args.workload != "pair":
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
