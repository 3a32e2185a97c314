"""GPU parity of the FP32-FMA path against the float64 oracle.

Tolerances: potentials within 1e-4 max(C) after the same iteration count,
plan applications within 1e-3 relative L2 (element-wise comparisons).
"""
import numpy as np
import pytest

import oracle as orc
from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import WORKLOADS, make_inputs, random_cloud
from tests.gpu_util import APPLY_TOL, F_TOL_FMA, max_abs, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


def _solve_both(inp, eps, iters, path="fma", splits=0):
    t = to_dev(inp)
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, iters, path=path, splits=splits)
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, iters)
    return np64(f), np64(g), fr, gr, C, t


@pytest.mark.parametrize("n,m,d", [(1, 1, 1), (1, 9, 2), (7, 1, 3), (33, 129, 3), (129, 33, 5),
                                   (1000, 1500, 2), (1500, 1000, 8), (700, 900, 16),
                                   (1025, 1023, 3)])
def test_ragged_shapes_match_oracle(n, m, d):
    inp = random_cloud(n, m, d, seed=100 + n + d, weights="lognormal")
    f, g, fr, gr, C, _ = _solve_both(inp, 0.1, 10)
    tol = F_TOL_FMA * C.max()
    assert max_abs(f, fr) <= tol
    assert max_abs(g, gr) <= tol


@pytest.mark.parametrize("splits", [1, 3, 17])
def test_forced_splits_agree(splits):
    inp = random_cloud(1300, 1100, 3, seed=7)
    f, g, fr, gr, C, _ = _solve_both(inp, 0.05, 20, splits=splits)
    assert max_abs(f, fr) <= F_TOL_FMA * C.max()
    assert max_abs(g, gr) <= F_TOL_FMA * C.max()


def test_c1_full_config():
    w = WORKLOADS["c1_n512_d2"]
    inp = make_inputs(w.name)
    eps, iters = w.stages[0]
    f, g, fr, gr, C, _ = _solve_both(inp, eps, iters)
    assert max_abs(f, fr) <= F_TOL_FMA * C.max()
    assert max_abs(g, gr) <= F_TOL_FMA * C.max()


def test_c2_reduced_solve_and_barycentric():
    w = WORKLOADS["c2_n10k_d3"]
    inp = make_inputs(w.name, n=3001, m=2999)
    eps, iters = w.stages[0]
    f, g, fr, gr, C, t = _solve_both(inp, eps, iters)
    assert max_abs(f, fr) <= F_TOL_FMA * C.max()
    assert max_abs(g, gr) <= F_TOL_FMA * C.max()
    T = fs.fs_barycentric(t["X"], t["a"], t["Y"], t["b"], eps, t["X"].new_tensor(fr),
                          t["Y"].new_tensor(gr))
    Tr = orc.barycentric(C, inp["a"], inp["b"], eps, fr.astype(np.float32), gr.astype(np.float32),
                         inp["Y"])
    assert rel_l2(np64(T), Tr) <= APPLY_TOL


def test_c2_full_config_solve_and_barycentric():
    """The full 10k x 10k, d = 3, eps = 0.01, 200-iteration workload, element-wise."""
    w = WORKLOADS["c2_n10k_d3"]
    inp = make_inputs(w.name)
    eps, iters = w.stages[0]
    f, g, fr, gr, C, t = _solve_both(inp, eps, iters, path="auto")
    assert max_abs(f, fr) <= F_TOL_FMA * C.max()
    assert max_abs(g, gr) <= F_TOL_FMA * C.max()
    T = fs.fs_barycentric(t["X"], t["a"], t["Y"], t["b"], eps, t["X"].new_tensor(f),
                          t["Y"].new_tensor(g))
    Tr = orc.barycentric(C, inp["a"], inp["b"], eps, f.astype(np.float32), g.astype(np.float32),
                         inp["Y"])
    assert rel_l2(np64(T), Tr) <= APPLY_TOL


@pytest.mark.parametrize("k", [1, 3, 4, 5, 16, 17, 40])
def test_apply_plan_matches_oracle(k):
    inp = random_cloud(900, 1300, 3, seed=50 + k, weights="lognormal")
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], 0.1, 5)
    f32, g32 = fr.astype(np.float32), gr.astype(np.float32)
    V = np.random.default_rng(k).standard_normal((1300, k)).astype(np.float32)
    t = to_dev(dict(inp, V=V, f=f32, g=g32))
    out = fs.fs_apply_plan(t["X"], t["a"], t["Y"], t["b"], 0.1, t["f"], t["g"], t["V"])
    ref = orc.apply_plan(C, inp["a"], inp["b"], 0.1, f32, g32, V)
    assert rel_l2(np64(out), ref) <= APPLY_TOL


def test_grad_x_matches_oracle():
    inp = random_cloud(800, 700, 2, seed=61, weights="lognormal")
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], 0.05, 50)
    f32, g32 = fr.astype(np.float32), gr.astype(np.float32)
    t = to_dev(dict(inp, f=f32, g=g32))
    out = fs.fs_grad_x(t["X"], t["a"], t["Y"], t["b"], 0.05, t["f"], t["g"])
    ref = orc.grad_x(C, inp["X"], inp["a"], inp["b"], 0.05, f32, g32, inp["Y"])
    assert rel_l2(np64(out), ref) <= APPLY_TOL


def test_host_buffers_give_the_device_result():
    inp = random_cloud(1200, 1000, 3, seed=70)
    t = to_dev(inp)
    fd, gd = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.05, 15)
    fh, gh = fs.fs_sinkhorn_solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.05, 15)
    assert isinstance(fh, np.ndarray)
    np.testing.assert_array_equal(np64(fd), fh.astype(np.float64))
    np.testing.assert_array_equal(np64(gd), gh.astype(np.float64))
    import torch
    pinned = {k: torch.from_numpy(v).pin_memory() for k, v in inp.items()}
    fp, gp = fs.fs_sinkhorn_solve(pinned["X"], pinned["a"], pinned["Y"], pinned["b"], 0.05, 15)
    np.testing.assert_array_equal(np64(fd), np64(fp))


def test_bitwise_deterministic():
    inp = random_cloud(2000, 1800, 3, seed=71)
    t = to_dev(inp)
    f1, g1 = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.02, 30)
    f2, g2 = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.02, 30)
    assert np.array_equal(np64(f1), np64(f2)) and np.array_equal(np64(g1), np64(g2))


def test_column_marginal_after_g_update_via_transposed_apply():
    """Just after a g-update the plan's column sums equal b; applying P^T
    (roles swapped) to ones measures them on the GPU alone."""
    inp = random_cloud(1500, 1200, 3, seed=72, weights="lognormal")
    t = to_dev(inp)
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.05, 25)
    ones = t["X"].new_ones((1500, 1))
    col = fs.fs_apply_plan(t["Y"], t["b"], t["X"], t["a"], 0.05, g, f, ones)
    # base-2 scores reach |s| ~ 600 here; float32 rounds them to ~4e-5 (relative
    # error of each plan entry), and the row scale 2^{phi + M} adds as much again
    np.testing.assert_allclose(np64(col)[:, 0], inp["b"].astype(np.float64), rtol=2e-4)


def test_translation_invariance_far_shift():
    """A common shift of X and Y leaves f, g unchanged (the library centres)."""
    inp = random_cloud(1000, 1100, 3, seed=73)
    t0 = to_dev(inp)
    shifted = dict(inp, X=(inp["X"] + np.float32(1000.0)), Y=(inp["Y"] + np.float32(1000.0)))
    t1 = to_dev(shifted)
    f0, g0 = fs.fs_sinkhorn_solve(t0["X"], t0["a"], t0["Y"], t0["b"], 0.1, 10)
    f1, g1 = fs.fs_sinkhorn_solve(t1["X"], t1["a"], t1["Y"], t1["b"], 0.1, 10)
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(orc.cost(shifted["X"], shifted["Y"]), inp["a"], inp["b"], 0.1, 10)
    # the shifted float32 inputs themselves are only accurate to ~6e-5 at 1000
    assert max_abs(np64(f1), fr) <= 1e-3 * C.max()
    assert max_abs(np64(f0), np64(f1)) <= 1e-2 * C.max()


def test_warm_start_equals_longer_run():
    """10 + 10 warm-started iterations equal 20 in one call, up to the float32
    rounding of the bias rebuilt from g at the restart (|beta| <~ 600 here,
    so ~4e-5 in base-2 score units, i.e. ~1e-6 in f)."""
    inp = random_cloud(900, 800, 2, seed=74)
    t = to_dev(inp)
    f1, g1 = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.05, 20)
    f2, g2 = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.05, 10)
    f2, g2 = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.05, 10, f2, g2)
    cmax = orc.cost(inp["X"], inp["Y"]).max()
    assert max_abs(np64(f1), np64(f2)) <= 1e-5 * cmax
    assert max_abs(np64(g1), np64(g2)) <= 1e-5 * cmax


def test_nonfinite_check_reports():
    inp = random_cloud(100, 120, 2, seed=75)
    t = to_dev(inp)
    g = t["Y"].new_zeros(120)
    g[3] = float("nan")
    with pytest.raises(fs.FlashSinkhornError) as ei:
        fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.1, 2, None, g, check_finite=True)
    assert ei.value.status == fs.FS_ERR_NONFINITE
    fs.fs_check()


def test_full_size_d3_converged_update_on_sampled_rows():
    """n = m = 50,000, d = 3, in the benchmark's launch configuration: after
    the workload's 100 iterations, one more warm-started f-update equals the
    oracle's point-by-point f-update from the GPU's g on 48 sampled rows, and
    the barycentric projection equals the oracle's on those rows."""
    w = WORKLOADS["c2_n50k_d3"]
    inp = make_inputs(w.name)
    eps, iters = w.stages[0]
    t = to_dev(inp)
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, iters, path="auto")
    g_prev = np64(g)
    f1, _ = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, 1, f.clone(), g.clone(),
                                 path="auto")
    rows = np.random.default_rng(5).choice(w.n, 48, replace=False)
    rows[:2] = [0, w.n - 1]
    ref = orc.f_update_rows(inp["X"], inp["Y"], inp["b"], eps, g_prev, rows)
    cmax = float(np.max(np.sum((inp["X"][rows, None, :].astype(np.float64)
                                - inp["Y"][None, :, :].astype(np.float64)) ** 2, axis=2)))
    assert max_abs(np64(f1)[rows], ref) <= F_TOL_FMA * cmax
    T = fs.fs_barycentric(t["X"], t["a"], t["Y"], t["b"], eps, f, g)
    f32, g32 = np64(f).astype(np.float32), g_prev.astype(np.float32)
    PY = orc.apply_plan_rows(inp["X"], inp["a"], inp["Y"], inp["b"], eps, f32, g32, inp["Y"], rows)
    Tr = PY / inp["a"][rows, None].astype(np.float64)
    assert rel_l2(np64(T)[rows], Tr) <= APPLY_TOL


@pytest.mark.parametrize("eps,iters", [(0.005, 6), (0.05, 12)])
def test_reference_offset_path_with_fixups(eps, iters):
    """n*m = 2^26 takes reference offsets after the first iterations; a cold
    start at small eps moves the LSEs by hundreds of log2 units between
    iterations, so many rows fail the guarded range and are recomputed by the
    fixup kernel.  The potentials must still match the oracle."""
    inp = make_inputs("c2_n10k_d3", n=8192, m=8192, seed=91)
    fs.fs_fixup_stats(reset=True)
    f, g, fr, gr, C, _ = _solve_both(inp, eps, iters, path="auto")
    launches, fixed = fs.fs_fixup_stats(reset=True)
    assert max_abs(f, fr) <= F_TOL_FMA * C.max()
    assert max_abs(g, gr) <= F_TOL_FMA * C.max()
    # one fixup pass per reference-offset half-update (this size runs as one launch)
    assert launches == 2 * (iters - 2)
    print(f"eps={eps}: {fixed} rows recomputed over {launches} fixup passes")


@pytest.mark.parametrize("d", [1, 2, 3])
def test_folded_offsets_match_the_oracle_and_do_not_depend_on_the_row_order(d):
    """From 2^28 score pairs on, a d <= 3 solve runs in Morton order with the
    row offsets folded into the staged columns (one affine fit per block of
    rows).  The whole 8-iteration solve equals the float64 oracle's element
    by element (f and g within 1e-4 max C); so does the solve of the same
    points with the caller's rows shuffled (the Morton order breaks ties of
    equal codes by the caller's order, so a block's rows, and its fit, can
    differ, but not beyond the tolerance).  d = 1 pads a zero coordinate,
    whose row of the fit's normal equations is zero but for the
    regularisation."""
    n = m = 16400                                    # n m = 2.69e8 >= 2^28
    inp = make_inputs("c2_n10k_d3", n=n, m=m, d=d, seed=404)
    eps, iters = 0.01, 8
    t = to_dev(inp)
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, iters)
    perm = np.random.default_rng(5).permutation(n)
    sh = dict(inp, X=np.ascontiguousarray(inp["X"][perm]), a=np.ascontiguousarray(inp["a"][perm]))
    ts = to_dev(sh)
    fs_, gs_ = fs.fs_sinkhorn_solve(ts["X"], ts["a"], ts["Y"], ts["b"], eps, iters)
    C = orc.cost(inp["X"], inp["Y"])                 # 2.15 GB of float64
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, iters)
    tol = F_TOL_FMA * C.max()
    del C
    assert max_abs(np64(f), fr) <= tol
    assert max_abs(np64(g), gr) <= tol
    assert max_abs(np64(fs_), fr[perm]) <= tol
    assert max_abs(np64(gs_), gr) <= tol
