"""Host-side logic of the multi-GPU benchmark, run as two gloo ranks on the
CPU: the max-over-ranks timing reduction, barriers, and the weak-scaling
aggregate (independent batches per rank, no data-path collective)."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, _ = bench.dist_env()
    dist = bench.init_dist(ws, "gloo")
    # per-rank kernel time differs; the job time is the slowest rank's
    local_ms = 100.0 + 50.0 * r
    mx = bench.reduce_max(dist, local_ms)
    bench.barrier(dist)
    value = bench.weak_scaling_value(ws, 1e9, 10, mx)
    q.put((r, mx, value))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_reduce_max_and_weak_scaling(world):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    expect_max = 100.0 + 50.0 * (world - 1)
    for r, mx, value in res:
        assert mx == expect_max
        # world ranks x 10 steps x 1 GFLOP in expect_max ms
        assert value == pytest.approx(world * 10 / (expect_max * 1e-3))


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(None, 3.5) == 3.5
    assert bench.weak_scaling_value(1, 2e9, 5, 1000.0) == pytest.approx(10.0)
