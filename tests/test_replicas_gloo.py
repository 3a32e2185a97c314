"""The N > 1 benchmark path on CPU: two gloo ranks exercise the host logic the
GPU replicas use (per-rank replica seeds, the max over ranks of the timed
region, the whole-job rate).  No GPU is involved."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from streaming_sinkhorn_solver_gb300.workloads import WORKLOADS, make_inputs
        w = WORKLOADS["c1_n512_d2"]
        seed = bench.replica_seed(w, rank)
        X = make_inputs(w.name, seed=seed)["X"]
        local_ms = 100.0 + 50.0 * rank            # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms)
        rate = bench.aggregate_rate(world, 1000.0, 4, total)
        q.put((rank, seed, float(X[0, 0]), total, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, x0, t0, v0), (r1, s1, x1, t1, v1) = res
    assert (r0, r1) == (0, 1)
    assert s1 == s0 + 1 and x0 != x1           # each rank solves its own replica
    assert t0 == t1 == 150.0                   # max over ranks
    assert v0 == v1 == pytest.approx(2 * 1000.0 * 4 / 0.150)


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate_rate(1, 10.0, 2, 1000.0) == pytest.approx(20.0)
