"""The multi-GPU path of bench.py is replicas only: every rank runs its own
layer and the job reports all ranks' tokens over the slowest rank's time.
These CPU tests run that bookkeeping as two gloo ranks (no GPU): the max over
ranks, the whole-job value, and the reference arm, which runs on rank 0 only."""
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


def _worker(rank, ws, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        t = bench.rank_max(1.0 + rank, ws, "cpu")   # rank 1 is the slow one
        v = bench.job_value(64 * 10, ws, t)
        assert bench._dist() == (ws, rank, rank)
        q.put((rank, t, v))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(ws))
    for rank, t, v in res:
        assert t == 2.0                       # max over ranks
        assert v == pytest.approx(2 * 640 / 2.0)  # all ranks' tokens / slowest time


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = type("A", (), dict(workload="tiny", tokens=4, steps=1, warmup=0))()
    assert bench.run_reference(args) is None
