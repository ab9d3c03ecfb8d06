"""The benchmark's multi-rank aggregation (barrier + max over ranks, sum of
work) on world_size 2 with the gloo backend on CPU: the path bench.py takes
under torchrun, minus the GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    local_ms = [3.0, 5.0][rank]
    out[rank] = bench.dist_max(local_ms, world, device="cpu")
    dist.destroy_process_group()


def test_two_rank_max_and_barrier():
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == 5.0 and out[1] == 5.0
