"""The benchmark's multi-rank host logic with two gloo ranks on the CPU: the
process group comes up from the torchrun environment variables, the timing
reduction returns the slowest rank's time on every rank, and the whole-job
rate counts every rank's units over that time (independent replicas, no data
collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    w, r, local = bench.dist_setup("gloo")
    assert (w, r, local) == (world, rank, rank)
    ms_local = 10.0 + 5.0 * rank          # rank 1 is the slow one
    ms_max = bench.max_over_ranks(w, ms_local)
    bench.barrier(w)
    rate = bench.whole_job_rate(w, 100.0, ms_max)
    out[rank] = (ms_max, rate)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        ms_max, rate = out[r]
        assert ms_max == pytest.approx(15.0)
        assert rate == pytest.approx(2 * 100.0 / 0.015)


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup("gloo") == (1, 0, 0)
    assert bench.max_over_ranks(1, 3.5) == 3.5
    assert bench.whole_job_rate(1, 8.0, 2.0) == pytest.approx(4000.0)
