"""The multi-GPU form of the path is replicas only (independent units, no
exchange step): every rank runs the whole workload on its own GPU and the
bench takes the slowest rank's time.  These tests run that host-side logic
as two gloo ranks on the CPU (no GPU, no kernel)."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench._rank_env()
    t_ms = bench.allreduce_max(10.0 + 5.0 * rank, w, "cpu")
    value = bench.job_value(w, 4096, 7, t_ms)
    dist.barrier()
    q.put((r, w, local, t_ms, value))
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    for r, w, local, t_ms, value in results:
        assert w == 2 and local == r
        assert t_ms == 15.0  # the slower rank's time, on every rank
        assert value == pytest.approx(2 * 4096 * 7 / 15e-3)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allreduce_max(3.5, 1, "cpu") == 3.5
    assert bench.job_value(1, 4096, 2, 1.0) == pytest.approx(4096 * 2 / 1e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from wavelet_guided_sparse_gb300 import workloads as wl
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), {"steps": 1, "warmup": 3})()
    assert bench.run_reference(args, wl.CONFIGS["tiny"]) == 0
    assert capsys.readouterr().out == ""  # no work and no line on rank 1
