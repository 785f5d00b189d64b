"""The benchmark's multi-rank host logic on CPU: two gloo ranks (no GPU).

With N > 1 every rank runs an independent replica of the workload; the only
cross-rank steps are the max-over-ranks time and the whole-job rate.  The
reference arm runs on rank 0 only; other ranks exit without work.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.dist_max(10.0 + rank)  # rank 1 is the slow one
    rate = bench.job_throughput(1000.0, world, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, rate))


def test_two_gloo_ranks_max_and_job_rate():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [11.0, 11.0]          # both ranks see the slowest time
    assert all(abs(r[2] - 2000.0 / 11e-3) < 1e-6 for r in res)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.5) == 3.5
    assert bench.job_throughput(10.0, 1, 2.0) == 5000.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    class A:
        impl, workload, steps, warmup = "reference", 5, 1, 0
    assert bench.run_reference(A()) is None  # returns immediately, prints nothing


def test_reference_arm_line_on_rank_0(monkeypatch, capsys):
    """Rank 0 prints one JSON line with the contract's keys: the oracle timed on the host cores
    on a sample of the workload (here the tiny fp32 one, so that the pass is instant)."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)

    class A:
        impl, workload, steps, warmup = "reference", 1, 2, 1
    bench.run_reference(A())
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] == 1 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
