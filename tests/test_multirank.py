"""The bench's N-GPU mode runs independent replicas (the SpMV path needs no
collective); its host logic -- barrier, max-over-ranks of the elapsed time,
whole-job throughput -- is checked here with two gloo ranks on the CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        elapsed = 10.0 + 5.0 * rank  # ms; rank 1 is the slowest
        got = bench.allreduce_max(elapsed, world, torch.device("cpu"))
        bytes_per_rank = 1_000_000_000
        value = world * bytes_per_rank / (got * 1e-3) / 1e9
        out[rank] = (got, value)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # whole-job throughput counts both replicas' work over the slowest rank
    assert abs(res[0][1] - 2 * 1.0 / 0.015) < 1e-9
