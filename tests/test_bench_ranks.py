"""The multi-rank parts of bench.py on CPU: two gloo ranks agree on the slowest
rank's time and on the whole-job rate (replicas, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    w, r, loc = bench.dist_env()
    assert (w, r, loc) == (world, rank, rank)
    bench.barrier(world)
    my_seconds = 1.0 + rank  # rank 1 is the slower one
    sec = bench.max_over_ranks(my_seconds, world)
    rate = bench.whole_job_rate(1000, 10, world, sec)
    out[rank] = (sec, rate)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_rate():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn",
                       join=True)
    assert out[0] == out[1]
    sec, rate = out[0]
    assert sec == 2.0
    assert rate == pytest.approx(1000 * 10 * 2 / 2.0)


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(10, 4, 1, 2.0) == 20.0
    args = bench.parse_args([])
    assert args.gpus == 1 and args.impl == "ours" and args.config == "shard175b"
    assert args.warmup >= 3
