"""The multi-GPU row split on two gloo ranks (CPU): each rank takes its
zig-zag chunks of one sequence, computes them with its inputs cut at the
chunk end (causality: a query row needs no later token) and must reproduce
the whole-sequence result for those rows; together the ranks cover every row
once.  The oracle stands in for each rank's GPU work."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import seeded_inputs as SI


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _layer(x, cfg, rows):
    from oracle import v4_oracle as O
    return O.attn_layer(cfg, x, rows=rows)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from sparse_compressed_attention_gb300 import rows as R
    from tests.helpers import inv_freq_for, oracle_inputs
    p = SI.preset("tiny_csa_f32", S=96)
    x = oracle_inputs(SI.make_layer_inputs(p, "cpu", seed=11, sink=True), inv_freq_for(p))
    cfg = dict(ratio=p["ratio"], overlap=p["overlap"], window=p["W"], topk=p["K"], rms_eps=1e-6,
               store_bf16=False)
    S = p["S"]
    cost = R.layer_cost(p["ratio"], p["K"], p["W"], heads=p["H"], dim=p["D"], idx_heads=p["Hi"], idx_dim=p["Di"])
    chunks = R.zigzag_chunks(S, world, rank, cost)
    whole = _layer(x, cfg, None)
    err = 0.0
    for a, b in chunks:
        # sequence-side inputs cut at b: the chunk's call sees only its prefix
        xc = {k: (v[:, :b] if isinstance(v, np.ndarray) and v.ndim >= 2 and v.shape[:2] == (p["B"], S) else v)
              for k, v in x.items()}
        part = _layer(xc, cfg, np.arange(a, b))
        err = max(err, float(np.abs(part["o"] - whole["o"][:, a:b]).max()),
                  float(np.abs(part["idx"] - whole["idx"][:, a:b]).max()))
    counts = torch.zeros(S, dtype=torch.int64)
    for a, b in chunks:
        counts[a:b] += 1
    dist.all_reduce(counts)
    out[rank] = (err, counts.tolist(), chunks)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_split_one_sequence_by_rows():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    for r in range(2):
        err, counts, chunks = out[r]
        assert err == 0.0, (r, err)
        assert counts == [1] * 96
        assert len(chunks) == 2
