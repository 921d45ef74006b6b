"""bench.py's multi-rank glue (barrier, max over ranks, whole-job throughput) with two gloo
ranks on the CPU: every rank runs the same per-GPU work, nothing on the data path is exchanged,
and rank 0 reports N x work / slowest rank time."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, w, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    ms = 10.0 + 5.0 * r            # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, w)
    work = 1.0e12                 # flops per rank per step
    value = w * work / (worst * 1e-3) / 1e12
    q.put((r, worst, value))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    assert [o[1] for o in out] == [15.0, 15.0]
    assert out[0][2] == pytest.approx(2 * 1.0e12 / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
