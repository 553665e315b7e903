"""bench.py's multi-rank host logic on CPU with the gloo backend and two
ranks (replicas, no data-path collective): every rank sees the slowest
rank's time, the whole-job value counts every rank's work over that time,
and the reference arm leaves ranks other than 0 without work."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, l = bench.dist_env()
    slowest = bench.reduce_max(1.5 + rank, w, device="cpu")
    value = bench.job_tflops(2e12, slowest, w)
    out.put((r, w, l, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_whole_job_value():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    for rank, (r, w, l, slowest, value) in enumerate(got):
        assert (r, w, l) == (rank, 2, rank)
        assert slowest == 2.5                 # max over ranks, on every rank
        assert value == pytest.approx(2e12 * 2 / 2.5e-3 / 1e12)


def test_reference_arm_leaves_other_ranks_idle(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    # returns before touching the oracle or any workload
    assert bench.run_reference(None, None) == 0


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    assert bench.job_tflops(1e9, 1.0, 1) == pytest.approx(1.0)   # 1 GFLOP in 1 ms
