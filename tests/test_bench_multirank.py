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


def test_crossover_summary_finds_the_first_m_from_which_w8a8_stays_faster():
    import bench

    rows = []
    for M, t4, t8 in [(1, 10.0, 15.0), (16, 14.0, 18.0), (32, 20.0, 19.0), (64, 18.0, 21.0), (128, 30.0, 25.0),
                      (256, 40.0, 30.0)]:
        rows.append({"K": 4096, "N": 14336, "M": M, "variant": "w4", "us": t4})
        rows.append({"K": 4096, "N": 14336, "M": M, "variant": "w8", "us": t8 - 1.0, "quant_us": 1.0})
    out = bench.crossover_summary(rows, 1900.0, 3800.0, 6800.0)["crossover"][0]
    assert out["measured_M"] == 128  # 32 is not the crossover: W4A16 wins again at 64
    assert out["measured_us"]["32"] == [20.0, 19.0]
    # the roofline crossover with FP8 at twice the BF16 rate sits near P16 / (2 BW)
    assert abs(out["roofline_M_gemm_only"] - out["simplified_P16_over_2BW"]) < 0.15 * out["simplified_P16_over_2BW"]
