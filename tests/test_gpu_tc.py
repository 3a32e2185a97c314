"""GPU parity of the tcgen05 tensor-core path against the float64 oracle.

Potentials must match within 1e-3 max(C) after the same iterations; plan
applications within 1e-3 relative L2.  Reduced sizes are compared element by
element; the full-size workloads, in the launch configuration the benchmark
uses, are compared on sampled rows the oracle evaluates one by one.
"""
import numpy as np
import pytest
from scipy.spatial.distance import cdist

import oracle as orc
from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import WORKLOADS, make_inputs, random_cloud
from tests.gpu_util import APPLY_TOL, F_TOL_TENSOR, max_abs, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


def _solve(inp, stages, path="tensor", splits=0):
    t = to_dev(inp)
    f = g = None
    for eps, it in stages:
        f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, it, f, g, path=path,
                                    splits=splits)
    return np64(f), np64(g), t


@pytest.mark.parametrize("n,m,d", [(1, 1, 17), (5, 300, 32), (129, 127, 64), (300, 260, 64),
                                   (257, 383, 100), (200, 300, 512), (130, 140, 600),
                                   (150, 129, 1024)])
def test_ragged_shapes_match_oracle(n, m, d):
    inp = random_cloud(n, m, d, seed=200 + n + d, spread=1.0 / np.sqrt(d), weights="lognormal")
    C = orc.cost(inp["X"], inp["Y"])
    eps = 0.05 * C.max()
    f, g, _ = _solve(inp, [(eps, 10)])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, 10)
    assert max_abs(f, fr) <= F_TOL_TENSOR * C.max()
    assert max_abs(g, gr) <= F_TOL_TENSOR * C.max()


@pytest.mark.parametrize("splits", [1, 2, 5])
def test_forced_splits(splits):
    inp = random_cloud(700, 900, 64, seed=9, spread=0.125)
    C = orc.cost(inp["X"], inp["Y"])
    f, g, _ = _solve(inp, [(0.1, 20)], splits=splits)
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], 0.1, 20)
    assert max_abs(f, fr) <= F_TOL_TENSOR * C.max()
    assert max_abs(g, gr) <= F_TOL_TENSOR * C.max()


def test_small_d_through_tensor_path_agrees_with_fma_path():
    inp = random_cloud(600, 500, 3, seed=10)
    C = orc.cost(inp["X"], inp["Y"])
    ft, gt, _ = _solve(inp, [(0.1, 15)], path="tensor")
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], 0.1, 15)
    assert max_abs(ft, fr) <= F_TOL_TENSOR * C.max()


@pytest.mark.parametrize("name,n,m", [("c3_n50k_d64", 2500, 2300), ("c4_n50k_d512", 1500, 1400),
                                      ("c5_n20k_m30k_d1024", 700, 1000)])
def test_config_recipes_reduced_full_schedule(name, n, m):
    """Each tensor-path workload's distributions and full eps schedule at a
    size the oracle finishes quickly (several tiles and a ragged tail)."""
    w = WORKLOADS[name]
    inp = make_inputs(name, n=n, m=m)
    C = orc.cost(inp["X"], inp["Y"])
    f, g, _ = _solve(inp, w.stages)
    fr, gr = orc.sinkhorn_stages(C, inp["a"], inp["b"], w.stages)
    assert max_abs(f, fr) <= F_TOL_TENSOR * C.max()
    assert max_abs(g, gr) <= F_TOL_TENSOR * C.max()


@pytest.mark.parametrize("name", ["c3_n50k_d64", "c4_n50k_d512", "c5_n20k_m30k_d1024"])
def test_full_size_first_update_on_sampled_rows(name):
    """Full-size workload, same launch configuration as the benchmark: after
    one iteration from g = 0, f on 48 sampled rows equals the oracle's
    point-by-point f-update."""
    w = WORKLOADS[name]
    inp = make_inputs(name)
    eps = w.stages[0][0]
    f, g, _ = _solve(inp, [(eps, 1)], path="auto")
    rows = np.random.default_rng(1).choice(w.n, 48, replace=False)
    rows[:2] = [0, w.n - 1]
    ref = orc.f_update_rows(inp["X"], inp["Y"], inp["b"], eps, np.zeros(w.m), rows)
    cmax = cdist(inp["X"][rows].astype(np.float64), inp["Y"].astype(np.float64), "sqeuclidean").max()
    assert max_abs(f[rows], ref) <= F_TOL_TENSOR * cmax
    assert np.isfinite(g).all()


def test_bitwise_deterministic_tensor():
    inp = random_cloud(1000, 1100, 64, seed=11, spread=0.125)
    f1, g1, _ = _solve(inp, [(0.05, 10)])
    f2, g2, _ = _solve(inp, [(0.05, 10)])
    assert np.array_equal(f1, f2) and np.array_equal(g1, g2)


def test_tensor_path_host_buffers():
    inp = random_cloud(500, 450, 96, seed=12, spread=0.1)
    fd, gd, _ = _solve(inp, [(0.05, 5)])
    fh, gh = fs.fs_sinkhorn_solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.05, 5, path="tensor")
    np.testing.assert_array_equal(fd, fh.astype(np.float64))
    np.testing.assert_array_equal(gd, gh.astype(np.float64))
