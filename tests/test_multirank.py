"""Replica mode of the benchmark across ranks, on CPU (gloo, world size 2):
each rank times its own replica; the job's throughput divides all ranks'
tokens by the slowest rank's time (max over ranks), with no data-path
collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    local = 0.5 + rank          # rank 1 is the slow one
    t = torch.tensor([local], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    agg = bench.aggregate([float(t.item())] * world, tokens_per_rank=128, steps=10)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, agg))


def test_two_rank_aggregation_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        assert res[r]["seconds"] == pytest.approx(1.5)
        assert res[r]["value"] == pytest.approx(2 * 128 * 10 / 1.5)
        assert res[r]["ms_per_step"] == pytest.approx(150.0)
