"""The benchmark's N > 1 path on CPU: two gloo ranks run independent
replicas and the job time is the slowest rank's (no data-path collective;
the QSA layer shards by sequence / query rows without any exchange)."""
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


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [120.0, 150.0][rank]
    job = bench.job_time_ms(ms, dist)
    val = bench.job_tokens_per_s(1000, world, job)
    dist.barrier()
    out.put((rank, job, val))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job, val in res:
        assert job == 150.0
        assert val == pytest.approx(2 * 1000 / 0.150)


def test_single_rank_is_identity():
    import bench

    assert bench.job_time_ms(42.0, None) == 42.0
    assert bench.job_tokens_per_s(10, 1, 1000.0) == 10.0


def test_oracle_sample_stays_bounded():
    """The CPU baseline's sample size: a per-row cost from two timed samples,
    falling back to the larger sample's average when the difference is tiny
    or negative (rows of unequal cost), and never above its cap."""
    import bench

    # a clean fit: 0.1 s fixed + 0.01 s per row, 12 s target
    assert bench.oracle_sample_rows([0.1 + 16 * 0.01, 0.1 + 32 * 0.01], 16, 10 ** 6, 12.0) in (1189, 1190)
    # the second sample came out faster than the first: bounded by the average
    n = bench.oracle_sample_rows([0.5, 0.45], 16, 10 ** 6, 12.0)
    assert 16 <= n <= 12.0 / (0.45 / 32) + 1
    # a tiny positive difference: the same fallback, and the cap holds
    assert bench.oracle_sample_rows([1.0, 1.0 + 1e-9], 16, 10 ** 6, 12.0) <= 12.0 / (1.0 / 32) + 1
    assert bench.oracle_sample_rows([1e-6, 2e-6], 16, 10 ** 6, 12.0) == 4096
    # never fewer than the calibration size, never more rows than there are
    assert bench.oracle_sample_rows([50.0, 100.0], 16, 10 ** 6, 12.0) == 16
    assert bench.oracle_sample_rows([0.01, 0.02], 16, 100, 12.0) == 100
