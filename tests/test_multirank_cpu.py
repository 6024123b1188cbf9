"""The N-GPU bench path runs independent replicas; its only cross-rank steps are a barrier
and a max of the per-rank times. Checked here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [120.0, 150.0][rank]  # rank 1 is the straggler
    slowest = bench.max_over_ranks(ms, world, device="cpu")
    dist.barrier()
    out[rank] = (slowest, bench.job_tflops(2.0e12, 10, slowest, world))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_the_work():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 150.0
    # 2 replicas x 10 steps x 2e12 FLOP over 0.15 s
    assert res[0][1] == pytest.approx(2 * 10 * 2.0e12 / 0.150 / 1e12)
    assert res[0][1] == res[1][1]


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_tflops(1e12, 4, 1000.0, 1) == pytest.approx(4.0)  # 4e12 FLOP in 1 s
