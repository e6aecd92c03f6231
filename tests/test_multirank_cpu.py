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


def test_reference_arm_under_torchrun():
    """`bench.py --impl reference` launched as the driver launches it for N > 1
    (torchrun, two ranks, 127.0.0.1), on the tiny workload: rank 0 times the
    oracle and prints one JSON line; the other rank exits 0 without work.  The
    reference arm needs no GPU, so its ranks form a gloo group."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--config", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "3", "--cpu-seconds", "0.1"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["extrapolated"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
