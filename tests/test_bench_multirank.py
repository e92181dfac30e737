"""The benchmark's multi-rank host logic on CPU with gloo (world size 2):
every rank runs its own replica; the job time is the slowest rank's, and the
value is the work of all ranks over that time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local = [3.0, 5.0][rank]          # this rank's timed region, ms
        mx = bench.max_over_ranks(local, dist, device="cpu")
        q.put((rank, mx, bench.job_tflops(world, 2e12, 10, mx)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_the_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(world))
    for rank, mx, value in out:
        assert mx == 5.0
        # 2 ranks x 10 steps x 2e12 FLOP in 5 ms = 8000 TFLOP/s
        assert value == pytest.approx(8000.0)


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks(4.2) == 4.2
    assert bench.job_tflops(1, 1e12, 2, 2.0) == pytest.approx(1000.0)
