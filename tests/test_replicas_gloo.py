"""The multi-GPU form of the benchmark is N independent replicas: no collective
on the data path, one max-over-ranks of the timed region, whole-job rates =
N x one replica's work / the slowest replica's time.  This runs that host logic
as two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = [120.0, 150.0][rank]          # rank 1 is the slower replica
        total = bench.max_over_ranks(local_ms)
        value, tok = bench.replica_rates(1000, 10, total, world)
        env = bench.dist_env()
        q.put((rank, total, value, tok, env))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, value, tok, env in got:
        assert total == 150.0                      # both ranks agree on the max
        assert env == (rank, world, rank)
        assert value == pytest.approx(2 * 1000 * 10 / 0.150 / 1e9)
        assert tok == pytest.approx(2 * 10 / 0.150)


def test_single_process_needs_no_group():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5
    v, t = bench.replica_rates(529821000, 100, 10.5, 1)
    assert t == pytest.approx(100 / 0.0105)
    assert v == pytest.approx(529821000 * 100 / 0.0105 / 1e9)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), {"reference_budget": 1.0, "steps": 1, "warmup": 3})()
    bench.run_reference(args)                      # returns at once, prints nothing
    assert capsys.readouterr().out == ""
