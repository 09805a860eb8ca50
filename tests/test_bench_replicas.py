"""The benchmark's multi-GPU accounting on the CPU: world-size-2 gloo ranks.

The path has no exchange step, so N GPUs run N independent replicas; the whole-job value is all
ranks' bytes over the slowest rank's time (the maximum over ranks, taken with an all-reduce), and
the oracle's reference arm runs on rank 0 only. Here two gloo processes stand in for the GPUs."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, local_ms, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        value, ms = bench.replica_throughput(1.0e9, 5, world, local_ms[rank])
        bench.barrier(world)
        q.put((rank, value, ms, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def _run(world, local_ms):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, local_ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_two_replicas_take_the_slowest_rank():
    out = _run(2, [10.0, 25.0])
    for rank, value, ms, env in out:
        assert ms == 25.0                                   # max over ranks, on every rank
        assert value == pytest.approx(2 * 5 * 1.0e9 / 25e-3 / 1e9)
        assert env == (2, rank, rank)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.replica_throughput(2.0e9, 4, 1, 8.0)
    assert ms == 8.0 and value == pytest.approx(2.0e9 * 4 / 8e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(steps=3, warmup=3, gpus=2)
    bench.run_reference(args)                               # rank 1: no work, no output
    assert capsys.readouterr().out == ""
