"""The multi-rank host path of bench.py on CPU (gloo, world size 2).

Each rank runs its own batch (weak scaling, no collective in the data path);
the only exchange is the maximum of the per-rank step times, and the
whole-job throughput is world x per-rank FLOPs / slowest time.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import synthetic_inputs as si
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = [1.0 + rank, 0.5 * (rank + 1), 2.0 - rank]
        got = bench.max_over_ranks(times, torch.device("cpu"), world)
        w = si.WORKLOADS[4]
        x = si.make_small(1, 1, 8, 64, seed=w.seed + bench.rank_seed_offset(rank))
        q.put((rank, got, dist.get_world_size(), bench.dist_env(), float(x["q"].float().sum())))
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_to_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, got, world, env, _ in res:
        assert world == 2
        assert got == [2.0, 1.0, 2.0]
        assert env == (2, rank, rank)
    # different ranks draw different batches
    assert res[0][4] != res[1][4]


def test_whole_job_throughput_is_weak_scaling():
    import bench
    one = bench.whole_job_tflops(1, 1e12, 10.0)
    assert one == pytest.approx(100.0)
    assert bench.whole_job_tflops(4, 1e12, 10.0) == pytest.approx(4 * one)
