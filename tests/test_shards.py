"""Row shards of the half-updates, without a GPU.

A half-update partitions by rows of the updated side (FlashSinkhorn,
Method 1: the f-update of row i needs only x_i and the whole other side), so
a G-GPU solve gives each GPU a range of rows and all-gathers the potential
after every half.  Here: the library's host partition (fs_shard_range, the
one its row-sharded solve launches by), and two gloo ranks that run the
float64 oracle's updates on their own rows, exchange them with an
all-gather, and reproduce the unsharded iteration bit for bit."""
import os
import socket

import numpy as np
import pytest

from streaming_sinkhorn_solver_gb300 import binding as fs


@pytest.fixture(scope="module")
def lib():
    from streaming_sinkhorn_solver_gb300.build import build
    build()
    return fs.load_library()


@pytest.mark.parametrize("rows,unit,shards", [
    (0, 256, 3), (1, 256, 1), (255, 256, 2), (256, 256, 2), (9000, 1024, 8), (8300, 256, 5),
    (8300, 256, 33), (8300, 256, 40), (2**31 - 1, 256, 7), (1000, 1, 1000)])
def test_partition_covers_every_row_once_on_unit_boundaries(lib, rows, unit, shards):
    ranges = [fs.fs_shard_range(rows, unit, shards, s) for s in range(shards)]
    assert ranges[0][0] == 0 and ranges[-1][1] == rows
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0                                  # contiguous, disjoint
    units = -(-rows // unit)
    sizes = []
    for r0, r1 in ranges:
        assert 0 <= r0 <= r1 <= rows
        assert r0 % unit == 0 or r0 == rows              # whole row blocks
        sizes.append(-(-(r1 - r0) // unit))
    assert sum(sizes) == units
    assert max(sizes) - min(sizes) <= 1                  # balanced to one unit
    if shards > units:
        assert sizes.count(0) == shards - units


def test_partition_rejects_bad_arguments(lib):
    for args in [(-1, 256, 2, 0), (10, 0, 2, 0), (10, 256, 0, 0), (10, 256, 2, 2),
                 (10, 256, 2, -1), (2**31, 256, 2, 0)]:
        with pytest.raises(fs.FlashSinkhornError):
            fs.fs_shard_range(*args)


def test_shard_units_are_the_row_blocks(lib):
    # the tensor kernels run 128-row tiles in CTA pairs: 256 rows
    assert fs.fs_shard_unit(64) == 256
    assert fs.fs_shard_unit(512) == 256
    assert fs.fs_shard_unit(3, "tensor") == 256
    # the FMA kernels: 256 threads x two rows per packed lane x row pairs
    for d in (1, 2, 3, 4, 8, 16):
        u = fs.fs_shard_unit(d)
        assert u % 512 == 0 and u >= 512
    with pytest.raises(fs.FlashSinkhornError):
        fs.fs_shard_unit(20, "fma")                      # beyond the FMA path
    with pytest.raises(fs.FlashSinkhornError):
        fs.fs_shard_unit(0)


# ---------------------------------------------------------------------------
# two gloo ranks: the exchange of a row-sharded solve, on the oracle

N, M, D, EPS, ITERS, UNIT = 300, 260, 3, 0.05, 4, 32


def _problem():
    rng = np.random.default_rng(1234)
    X = rng.random((N, D)).astype(np.float32)
    Y = (rng.random((M, D)) * 0.8 + 0.1).astype(np.float32)
    a = rng.dirichlet(np.ones(N)).astype(np.float32)
    b = rng.dirichlet(np.ones(M)).astype(np.float32)
    return X, a, Y, b


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _all_gather_rows(dist, torch, local: np.ndarray, ranges, rank: int) -> np.ndarray:
    """Every rank's rows, in rank order; gloo all_gather wants equal sizes, so
    each piece is padded to the longest range."""
    width = max(r1 - r0 for r0, r1 in ranges)
    buf = torch.zeros(width, dtype=torch.float64)
    buf[: len(local)] = torch.from_numpy(local)
    parts = [torch.zeros(width, dtype=torch.float64) for _ in ranges]
    dist.all_gather(parts, buf)
    return np.concatenate([parts[r][: r1 - r0].numpy() for r, (r0, r1) in enumerate(ranges)])


def _rank_main(rank: int, world: int, port: int, q):
    import torch
    import torch.distributed as dist
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, a, Y, b = _problem()
        C = oracle.cost(X, Y)
        xr = [fs.fs_shard_range(N, UNIT, world, s) for s in range(world)]
        yr = [fs.fs_shard_range(M, UNIT, world, s) for s in range(world)]
        (x0, x1), (y0, y1) = xr[rank], yr[rank]
        g = np.zeros(M)
        for _ in range(ITERS):
            f_loc = oracle.f_update(C[x0:x1], b, EPS, g)          # own rows, all of g
            f = _all_gather_rows(dist, torch, f_loc, xr, rank)
            g_loc = oracle.g_update(C[:, y0:y1], a, EPS, f)       # own columns, all of f
            g = _all_gather_rows(dist, torch, g_loc, yr, rank)
        q.put((rank, (x0, x1), (y0, y1), f.tobytes(), g.tobytes()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_unsharded_iteration():
    import oracle
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    del torch
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, xa, ya, f0, g0), (r1, xb, yb, f1, g1) = res
    assert (r0, r1) == (0, 1)
    assert xa[1] == xb[0] and ya[1] == yb[0]              # each rank its own rows
    assert xa[1] % UNIT == 0 and 0 < xa[1] < N
    assert f0 == f1 and g0 == g1                          # every rank holds the same potentials

    X, a, Y, b = _problem()
    C = oracle.cost(X, Y)
    g = np.zeros(M)
    for _ in range(ITERS):
        f = oracle.f_update(C, b, EPS, g)
        g = oracle.g_update(C, a, EPS, f)
    assert np.frombuffer(f0, np.float64).tobytes() == f.tobytes()
    assert np.frombuffer(g0, np.float64).tobytes() == g.tobytes()
    fo, go = oracle.sinkhorn(C, a, b, EPS, ITERS)
    np.testing.assert_allclose(f, fo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g, go, rtol=0, atol=1e-12)
