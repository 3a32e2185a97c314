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


# --- plan application on the tensor path ------------------------------------

def _potentials(inp, eps, iters):
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, iters)
    return C, fr.astype(np.float32), gr.astype(np.float32)


@pytest.mark.parametrize("n,m,d,k", [(300, 400, 64, 1), (257, 383, 64, 16), (129, 700, 32, 17),
                                     (400, 300, 100, 64), (200, 260, 512, 130),
                                     (150, 170, 600, 300), (140, 129, 1024, 64)])
def test_apply_plan_tensor_matches_oracle(n, m, d, k):
    inp = random_cloud(n, m, d, seed=300 + k + d, spread=1.0 / np.sqrt(d), weights="lognormal")
    C = orc.cost(inp["X"], inp["Y"])
    eps = 0.05 * C.max()
    _, f32, g32 = _potentials(inp, eps, 5)
    V = np.random.default_rng(k).standard_normal((m, k)).astype(np.float32)
    t = to_dev(dict(inp, V=V, f=f32, g=g32))
    out = fs.fs_apply_plan(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"], path="tensor")
    ref = orc.apply_plan(C, inp["a"], inp["b"], eps, f32, g32, V)
    assert rel_l2(np64(out), ref) <= APPLY_TOL


@pytest.mark.parametrize("d", [64, 512])
def test_grad_and_barycentric_tensor_match_oracle(d):
    inp = make_inputs("c4_n50k_d512", n=900, m=1000, d=d)
    C, f32, g32 = _potentials(inp, 0.05, 30)
    t = to_dev(dict(inp, f=f32, g=g32))
    grad = fs.fs_grad_x(t["X"], t["a"], t["Y"], t["b"], 0.05, t["f"], t["g"], path="tensor")
    ref = orc.grad_x(C, inp["X"], inp["a"], inp["b"], 0.05, f32, g32, inp["Y"])
    assert rel_l2(np64(grad), ref) <= APPLY_TOL
    T = fs.fs_barycentric(t["X"], t["a"], t["Y"], t["b"], 0.05, t["f"], t["g"], path="tensor")
    Tr = orc.barycentric(C, inp["a"], inp["b"], 0.05, f32, g32, inp["Y"])
    assert rel_l2(np64(T), Tr) <= APPLY_TOL


@pytest.mark.parametrize("splits", [1, 3])
def test_apply_forced_splits_wide_output_blocks(splits):
    """d >= 256 and more than 128 value columns: 256-column output blocks with
    one value slot, a ragged second block (k = 290 -> 256 + 48), several
    column tiles per CTA and split partials."""
    inp = random_cloud(300, 900, 300, seed=17, spread=1.0 / np.sqrt(300), weights="lognormal")
    C, f32, g32 = _potentials(inp, 0.05 * 2.0, 6)
    V = np.random.default_rng(5).standard_normal((900, 290)).astype(np.float32)
    t = to_dev(dict(inp, V=V, f=f32, g=g32))
    out = fs.fs_apply_plan(t["X"], t["a"], t["Y"], t["b"], 0.1, t["f"], t["g"], t["V"],
                           path="tensor", splits=splits)
    ref = orc.apply_plan(C, inp["a"], inp["b"], 0.1, f32, g32, V)
    assert rel_l2(np64(out), ref) <= APPLY_TOL


@pytest.mark.parametrize("splits", [1, 3])
def test_apply_forced_splits(splits):
    inp = random_cloud(500, 650, 64, seed=13, spread=0.125, weights="lognormal")
    C, f32, g32 = _potentials(inp, 0.1, 10)
    V = np.random.default_rng(2).standard_normal((650, 40)).astype(np.float32)
    t = to_dev(dict(inp, V=V, f=f32, g=g32))
    out = fs.fs_apply_plan(t["X"], t["a"], t["Y"], t["b"], 0.1, t["f"], t["g"], t["V"],
                           path="tensor", splits=splits)
    ref = orc.apply_plan(C, inp["a"], inp["b"], 0.1, f32, g32, V)
    assert rel_l2(np64(out), ref) <= APPLY_TOL


def test_column_marginal_tensor_path():
    """After a tensor-path solve, the last half-update (the g-update) makes
    the column sums equal b; the transposed apply measures them on the GPU."""
    inp = make_inputs("c3_n50k_d64", n=3000, m=2700)
    t = to_dev(inp)
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.1, 30, path="tensor")
    ones = t["X"].new_ones((3000, 1))
    col = fs.fs_apply_plan(t["Y"], t["b"], t["X"], t["a"], 0.1, g, f, ones, path="tensor")
    # fp16 plan entries (relative 2^-11 each) averaged over many rows
    assert rel_l2(np64(col)[:, 0], inp["b"]) <= APPLY_TOL


@pytest.mark.parametrize("name", ["c4_n50k_d512", "c5_n20k_m30k_d1024"])
def test_full_size_plan_application_on_sampled_rows(name):
    """Full-size workload: potentials from the oracle on 24 sampled rows (g = 0,
    f = the oracle's f-update there), the workload's plan operator on the GPU,
    compared with the oracle's point-by-point application on those rows."""
    w = WORKLOADS[name]
    inp = make_inputs(name)
    eps = w.stages[-1][0]
    rows = np.random.default_rng(3).choice(w.n, 24, replace=False)
    rows[:2] = [0, w.n - 1]
    g = np.zeros(w.m)
    fr = orc.f_update_rows(inp["X"], inp["Y"], inp["b"], eps, g, rows)
    f = np.zeros(w.n, np.float32)
    f[rows] = fr.astype(np.float32)
    V = inp["V"] if w.apply == "pv" else inp["Y"]
    t = to_dev(dict(inp, f=f, g=g.astype(np.float32)))
    if w.apply == "pv":
        out = fs.fs_apply_plan(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"])
        ref = orc.apply_plan_rows(inp["X"], inp["a"], inp["Y"], inp["b"], eps, f, g, V, rows)
    else:
        out = fs.fs_grad_x(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"])
        PY = orc.apply_plan_rows(inp["X"], inp["a"], inp["Y"], inp["b"], eps, f, g, V, rows)
        ref = 2.0 * (inp["a"][rows, None].astype(np.float64) * inp["X"][rows] - PY)
    assert rel_l2(np64(out)[rows], ref) <= APPLY_TOL


@pytest.mark.parametrize("d,eps,iters", [(64, 0.01, 6), (64, 0.1, 10), (256, 0.02, 6),
                                         (1024, 0.02, 6)])
def test_reference_offset_path_with_fixups(d, eps, iters):
    """n*m = 2^26 takes reference offsets after the first iterations (one-CTA
    kernel at d = 64, CTA pairs at d = 256, CTA pairs with Q streamed through
    the ring at d = 1024).  A cold start at small eps moves
    the LSEs far between iterations, so many rows fail the guarded range and
    are recomputed by the FP32 fixup; the potentials must still match."""
    inp = make_inputs("c3_n50k_d64", n=8192, m=8192, d=d, seed=93)
    C = orc.cost(inp["X"], inp["Y"])
    f, g, _ = _solve(inp, [(eps, iters)], path="auto")
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, iters)
    assert max_abs(f, fr) <= F_TOL_TENSOR * C.max()
    assert max_abs(g, gr) <= F_TOL_TENSOR * C.max()


@pytest.mark.parametrize("n,m,d,splits", [(8250, 8300, 40, 0), (8200, 8192, 100, 0),
                                          (8192, 8192, 128, 0), (8192, 8192, 64, 1),
                                          (8192, 8192, 64, 4), (8200, 8300, 1000, 1),
                                          (8300, 8200, 1000, 0)])
def test_reference_offset_kernel_shapes(n, m, d, splits):
    """The reference-offset kernels at n*m >= 2^26: the one-CTA kernel with
    one K chunk and zero-padded dimensions (d = 40), two chunks (d = 100,
    128), ragged row and column tiles, and forced column splits (1: the guard
    in the kernel itself; 4: the guard in the split merge); the CTA-pair
    kernel with Q streamed through the ring (d = 1000: 16 chunks, the last
    zero-padded) with ragged tiles, unsplit and split."""
    inp = make_inputs("c3_n50k_d64", n=n, m=m, d=d, seed=94 + d)
    C = orc.cost(inp["X"], inp["Y"])
    f, g, _ = _solve(inp, [(0.05, 6)], path="auto", splits=splits)
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], 0.05, 6)
    assert max_abs(f, fr) <= F_TOL_TENSOR * C.max()
    assert max_abs(g, gr) <= F_TOL_TENSOR * C.max()

