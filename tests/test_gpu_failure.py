"""Failure detection on the GPU without a fault: a bounded wait that runs out
reports FS_ERR_TIMEOUT through the device error word, and the context stays
usable (the next call still matches the oracle).  The wait is the same
inline-PTX loop the tensor-core kernels use; nothing traps, faults or hangs.
"""
import numpy as np
import pytest

import oracle as orc
from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import random_cloud
from tests.gpu_util import F_TOL_FMA, max_abs, np64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    fs.fs_check()                                   # start from a clear error word
    fs.fs_wait_selftest(2_000_000)                  # 2 ms deadline, nothing arrives
    with pytest.raises(fs.FlashSinkhornError) as e:
        fs.fs_check()
    assert e.value.status == fs.FS_ERR_TIMEOUT
    fs.fs_check()                                   # the word was cleared
    inp = random_cloud(300, 280, 3, seed=4)
    t = to_dev(inp)
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.1, 10)
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], 0.1, 10)
    assert max_abs(np64(f), fr) <= F_TOL_FMA * C.max()
    fs.fs_check()


@pytest.mark.parametrize("bad", [0, 999, 2_000_000_000])
def test_wait_selftest_rejects_deadlines_out_of_range(bad):
    with pytest.raises(fs.FlashSinkhornError) as e:
        fs.fs_wait_selftest(bad)
    assert e.value.status == fs.FS_ERR_INVALID_ARG


def test_grid_barrier_that_runs_out_reports_timeout_and_context_survives():
    """The one-launch solve's grid barrier: one of two co-resident blocks
    never arrives, the other's wait gives up after 2 ms."""
    fs.fs_check()
    fs.fs_barrier_selftest(2_000_000)
    with pytest.raises(fs.FlashSinkhornError) as e:
        fs.fs_check()
    assert e.value.status == fs.FS_ERR_TIMEOUT
    fs.fs_check()
    inp = random_cloud(400, 350, 2, seed=8)           # a one-launch solve right after
    t = to_dev(inp)
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.1, 10)
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], 0.1, 10)
    assert max_abs(np64(f), fr) <= F_TOL_FMA * C.max()
    assert max_abs(np64(g), gr) <= F_TOL_FMA * C.max()
    fs.fs_check()


@pytest.mark.parametrize("bad", [0, 999, 2_000_000_000])
def test_barrier_selftest_rejects_deadlines_out_of_range(bad):
    with pytest.raises(fs.FlashSinkhornError) as e:
        fs.fs_barrier_selftest(bad)
    assert e.value.status == fs.FS_ERR_INVALID_ARG
