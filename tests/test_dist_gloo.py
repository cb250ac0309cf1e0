"""Rank aggregation of the benchmark (max time, summed tokens) on two gloo
ranks on the CPU: the only cross-rank step of the multi-GPU run."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = (bench.max_over_ranks(10.0 + rank), bench.sum_over_ranks(1000.0 * (rank + 1)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_time_and_token_sum():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == (11.0, 3000.0) and out[1] == (11.0, 3000.0)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(5.0) == 5.0 and bench.sum_over_ranks(7.0) == 7.0
