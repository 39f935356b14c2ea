"""The benchmark's multi-rank logic on CPU: two gloo ranks, barrier, max over ranks.

Each rank of a multi-GPU run is an independent replica of the workload (weak
scaling); the only cross-rank steps are the barrier around the timed region
and the max of the elapsed times, exercised here without a GPU.
"""
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        slowest = bench.reduce_max(local_ms)
        bench.barrier()
        q.put((rank, slowest, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[1] for g in got] == [15.0, 15.0]
    assert [g[2] for g in got] == [(0, 0, 2), (1, 1, 2)]


def test_job_throughput_is_all_units_over_the_slowest_rank():
    assert bench.job_throughput(100.0, 2, 4.0) == 50.0
    assert bench.job_throughput(100.0, 1, 4.0) == 25.0


def test_reduce_max_without_process_group_is_identity():
    assert bench.reduce_max(3.5) == 3.5


def test_reference_arm_prints_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload, steps, warmup, weights = "ffn_down", 1, 3, "raw"
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
