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
