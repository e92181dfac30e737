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


def test_config_roofline_picks_the_binding_limit():
    import bench
    peaks = {"bf16_tflops": 1936.0, "hbm_gbs": 6786.9, "source": "measured"}
    # the headline: compute-bound
    r = bench.config_roofline("bf16", 8192, 8192, 8192, 600.0, peaks, 152, 2070.0)
    assert r["bound"] == "tensor" and r["tflops"] == pytest.approx(2 * 8192 ** 3 / 600e-6 / 1e12)
    assert r["frac"] == pytest.approx(r["tflops"] / 1936.0)
    # (8, 8192, 8192): 134.6 MB for 1.07 GFLOP -- HBM-bound
    r = bench.config_roofline("f16", 8, 8192, 8192, 25.0, peaks, 152, 2070.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["algorithmic_bytes"] == (8 * 8192 + 8192 * 8192) * 2 + 8 * 8192 * 4
    assert r["frac"] == pytest.approx(r["algorithmic_bytes"] / 25e-6 / 1e9 / 6786.9)
    # (16384, 128, 4096) is HBM-bound too; (4000, 3000, 1000) is not
    assert bench.config_roofline("f16", 16384, 128, 4096, 27.0, peaks, 152, 2070.0)["bound"] == "hbm"
    assert bench.config_roofline("f16", 4000, 3000, 1000, 30.0, peaks, 152, 2070.0)["bound"] == "tensor"
    # FP32 on the CUDA cores: 152 SMs x 256 FLOP/clk at the sampled clock
    r = bench.config_roofline("f32", 4096, 4096, 4096, 2000.0, peaks, 152, 2000.0)
    assert r["bound"] == "alu" and r["peak"] == pytest.approx(152 * 256 * 2.0e9 / 1e12)


def test_clock_bins_and_clock_limited_peak():
    import bench
    assert bench.clock_limited_tflops(152, 8192, 2070.0) == pytest.approx(2577.6, rel=1e-4)
    bins = bench.bin_by_clock([(1800.0, [1900.0, 1905.0, 1900.0]), (1700.0, [1800.0]),
                               (1820.0, [1900.0]), (1000.0, [])])
    assert bins == [{"sm_mhz": 1800.0, "tflops": 1700.0, "chunks": 1},
                    {"sm_mhz": 1900.0, "tflops": 1810.0, "chunks": 2}]


def test_output_samples_cover_first_middle_last_rows():
    import numpy as np
    import bench
    C = np.arange(100 * 7, dtype=np.float32).reshape(100, 7)
    smp = bench.output_samples(C, 100, 7, seed=1, band=4, n_entries=16)
    assert smp["rows"] == [0, 1, 2, 3, 50, 51, 52, 53, 96, 97, 98, 99]
    assert np.array_equal(smp["row_values"], C[smp["rows"]])
    assert np.array_equal(smp["entry_values"], C[smp["entry_rows"], smp["entry_cols"]])
    assert (smp["entry_cols"][:4] == 6 - np.arange(4)).all()
    tiny = bench.output_samples(C[:3], 3, 7, seed=1, band=8, n_entries=8)
    assert tiny["rows"] == [0, 1, 2]
