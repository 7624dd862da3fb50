"""Replica path of the benchmark (one process per GPU, no data-path collective), exercised on CPU
with the gloo backend and two ranks: the max-over-ranks timing and the whole-job throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = 10.0 + 5.0 * rank          # rank 1 is the slowest replica
        m = bench.max_over_ranks(ms)
        out[rank] = (m, bench.replica_tokens_per_s(world, 50, 4, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == pytest.approx(15.0)
    # 2 replicas x 50 steps x 4 tokens in 15 ms
    assert res[0][1] == pytest.approx(2 * 50 * 4 / 15e-3)


def test_single_process_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
