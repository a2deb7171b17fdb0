"""The N-replica path of bench.py: one process per GPU, each running the whole
product on its own copy of the workload (the path has no exchange step); the
job's time is the slowest rank's, its throughput the bytes of all ranks.
Checked here with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, ws: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench

    ms_local = [0.30, 0.45][rank]
    t_max, value = bench.aggregate(ms_local, 1_000_000, ws, torch.device("cpu"))
    q.put((rank, t_max, value))
    dist.destroy_process_group()


def test_two_replicas_report_slowest_rank_and_total_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, value in got:
        assert t_max == pytest.approx(0.45)
        assert value == pytest.approx(2 * 1_000_000 / 0.45e-3 / 1e9)


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    t_max, value = bench.aggregate(0.5, 2_000_000, 1, torch.device("cpu"))
    assert t_max == 0.5 and value == pytest.approx(4.0)
