"""The multi-GPU bench harness logic on CPU: two gloo ranks (replicas only,
no data-path collective) agree on the slowest rank's time, and the whole-job
value counts every replica's bytes."""

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


def _worker(rank, world, port, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        dist.barrier()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
        out[rank] = (slowest, bench.job_throughput(1_000_000_000, 4, w, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == pytest.approx(15.0) and res[1][0] == pytest.approx(15.0)
    # 2 replicas x 4 steps x 1 GB in 15 ms
    assert res[0][1] == pytest.approx(2 * 4 * 1.0 / 0.015)


def test_clock_summary_flags_throttle_reasons():
    import bench

    lines = ["0, 1900, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
             "0, 1950, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage"]
    c = bench.summarize_clocks(lines)
    assert c["sm_mhz"] == pytest.approx(1925.0) and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 2
    assert bench.summarize_clocks([]) is None
