"""The N > 1 path is replicas only: independent decodes, one per GPU, timed
between barriers and reduced with MAX over ranks.  Its host logic runs here
as two gloo ranks on CPU (no GPU): both ranks see the slowest rank's time,
the job's throughput counts every replica's bytes, and the reference arm
does its work on rank 0 only."""

import contextlib
import io
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.replica_env()
        ms = bench.max_over_ranks(times[rank], w, "cpu")
        dist.barrier()
        out.put((r, local, w, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, times = 2, [1.25, 1.75]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1] and [g[1] for g in got] == [0, 1]
    assert all(g[2] == world for g in got)
    assert all(g[3] == max(times) for g in got)


def test_job_throughput_counts_every_replica():
    import bench
    # two replicas moving 3.6 GB each per 1.5 ms unit: 4.8 TB/s for the job
    assert bench.job_gbs(3.6e9, 1.5, 2) == pytest.approx(4800.0)
    assert bench.job_gbs(3.6e9, 1.5, 1) == pytest.approx(2400.0)
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5


def test_reference_arm_works_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(None)       # rank 1 returns before reading any argument
    assert buf.getvalue() == ""
