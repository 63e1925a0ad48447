"""Host logic of bench.py's multi-rank run, on CPU with the gloo backend: every rank runs a
full replica of the workload, the job's step time is the maximum over ranks, and only rank
0 prints (and only rank 0 times the oracle)."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    try:
        w, r, loc = bench.dist_setup()
        dist.init_process_group("gloo", rank=r, world_size=w)
        ms = bench.max_over_ranks(1.0 + 0.5 * r, w, torch.device("cpu"))
        # rank != 0 leaves the reference arm without timing anything or printing
        class A:
            steps, warmup, gpus = 1, 0, w
        buf = io.StringIO()
        if r != 0:
            with redirect_stdout(buf):
                bench.run_reference(A, w, r)
        dist.barrier()
        dist.destroy_process_group()
        q.put((r, w, loc, ms, buf.getvalue()))
    except Exception as e:  # reported to the parent
        q.put((rank, "error", repr(e)))


def test_two_gloo_ranks_max_and_silence():
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for item in res:
        assert item[1] != "error", item
    by_rank = {item[0]: item for item in res}
    assert sorted(by_rank) == [0, 1]
    for r, (rr, w, loc, ms, out) in by_rank.items():
        assert (rr, w, loc) == (r, world, r)
        assert ms == pytest.approx(1.5)  # the slowest rank's time on every rank
    assert by_rank[1][4] == ""


def test_job_throughput_counts_all_replicas():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_gbs(10**9, 1, 1.0)
    assert one == pytest.approx(1000.0)
    assert bench.job_gbs(10**9, 4, 1.0) == pytest.approx(4 * one)
    assert bench.job_gbs(10**9, 4, 2.0) == pytest.approx(2 * one)


def test_dist_setup_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (1, 0, 0)
