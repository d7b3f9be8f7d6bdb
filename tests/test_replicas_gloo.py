"""The benchmark's multi-GPU mode (N independent replicas) on the CPU with
world_size-2 gloo ranks: the job time is the slowest rank's, the whole-job
throughput counts every rank's units, and the reference arm runs on rank 0
only (the other ranks exit at once, without work)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [40.0, 55.0][rank]
        job_ms = bench.max_over_ranks(local_ms)
        gbs = bench.whole_job_gbs(world, 10, 1_000_000_000, job_ms)
        dist.barrier()
        q.put((rank, job_ms, gbs))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for _, job_ms, gbs in res:
        assert job_ms == 55.0                               # the slowest rank
        assert gbs == pytest.approx(2 * 10 * 1.0 / 0.055)    # all ranks' bytes / slowest time


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.whole_job_gbs(1, 4, 2_000_000_000, 1000.0) == pytest.approx(8.0)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "host_inputs", lambda *a, **k: called.append(1))
    bench.run_reference(argparse.Namespace(steps=5, warmup=3, gpus=2))
    assert called == [] and capsys.readouterr().out == ""
