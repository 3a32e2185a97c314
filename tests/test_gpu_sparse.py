"""GPU parity of the block-sparse low-dimensional solver against the float64
oracle (``oracle/block_sparse.py``), through the C ABI.

Source: "FlashSinkhorn 2: Block-Sparse Entropic Optimal Transport" (patty.io
post).  Bars:
* Morton order: integer work, bit-exact.
* Screening: a decision is compared where the oracle's float64 bound is at
  least 0.02 log2 units from the threshold (the GPU evaluates it in float32);
  the kept lists must be strictly increasing.
* Potentials: within 1e-4 max(C) of the oracle after the same schedule (the
  FP32-FMA tolerance); a borderline block kept on one side and not the other
  changes a marginal by less than tau of its block's weight.
* Full size: dense column marginals at the returned potentials lie in
  [b_j, b_j + tau W_J] (the screening guarantee), checked on sampled columns.
"""
import numpy as np
import pytest

import oracle as orc
import oracle.block_sparse as bsp
from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import (WORKLOADS, clustered_cloud, make_inputs,
                                                       random_cloud)
from tests.gpu_util import F_TOL_FMA, max_abs, np64, to_dev

pytestmark = pytest.mark.gpu

MARGIN = 0.02


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


def _lattice(n, d, seed):
    rng = np.random.default_rng(seed)
    P = rng.integers(0, 50, size=(n, d)).astype(np.float32) * np.float32(0.37)
    P[: n // 3] = P[n // 3: 2 * (n // 3)]          # exact duplicates: ties keep input order
    return P


@pytest.mark.parametrize("n,m,d", [(1, 1, 1), (5, 300, 2), (1000, 777, 3), (5000, 4100, 3),
                                   (4099, 2048, 1), (3000, 3001, 2),
                                   # above d = 3: floor(63 / d) bits per axis
                                   (1000, 900, 4), (3000, 2000, 5), (7, 1, 6), (2000, 2100, 8)])
def test_morton_order_bit_exact(n, m, d):
    c = random_cloud(n, m, d, seed=n + m + d)
    t = to_dev(c)
    px, py = fs.fs_morton_order(t["X"], t["Y"])
    ox, oy = bsp.morton_order(c["X"], c["Y"])
    np.testing.assert_array_equal(px.cpu().numpy(), ox)
    np.testing.assert_array_equal(py.cpu().numpy(), oy)


@pytest.mark.parametrize("d", [1, 2, 3, 4, 8])
def test_morton_order_with_ties_bit_exact(d):
    X, Y = _lattice(3000, d, 1), _lattice(2100, d, 2)
    import torch
    px, py = fs.fs_morton_order(torch.from_numpy(X).cuda(), torch.from_numpy(Y).cuda())
    ox, oy = bsp.morton_order(X, Y)
    np.testing.assert_array_equal(px.cpu().numpy(), ox)
    np.testing.assert_array_equal(py.cpu().numpy(), oy)


def _screen_case(name, n, m, d, eps, dense_iters):
    if name == "clustered":
        # 12 clusters of standard deviation 0.03 in [0, 1]^d
        inp = clustered_cloud(n, m, d, 12, 0.03, seed=n + d)
    else:
        inp = make_inputs(name, n=n, m=m, d=d)
    if n * m > 5e7:
        # one iteration from g = 0, row by row (no n x m cost matrix)
        f = orc.f_update_rows(inp["X"], inp["Y"], inp["b"], eps, np.zeros(m), np.arange(n))
        g = orc.f_update_rows(inp["Y"], inp["X"], inp["a"], eps, f, np.arange(m))
        return inp, f.astype(np.float32), g.astype(np.float32)
    C = orc.cost(inp["X"], inp["Y"])
    f, g = orc.sinkhorn(C, inp["a"], inp["b"], eps, dense_iters)
    return inp, f.astype(np.float32), g.astype(np.float32)


@pytest.mark.parametrize("name,n,m,d,eps,tau,side", [
    ("c2_n10k_d3", 3000, 2500, 3, 0.003, 1e-4, 0),
    ("c2_n10k_d3", 3000, 2500, 3, 0.003, 1e-4, 1),
    ("c2_n10k_d3", 4000, 4000, 2, 0.001, 1e-6, 0),
    ("c1_n512_d2", 2600, 1900, 2, 0.02, 1e-3, 1),
    ("c2_n10k_d3", 2000, 2200, 1, 0.0005, 1e-5, 0),
    # 157 x 141 blocks: the two-level cull (super-blocks of 16 blocks) runs
    ("c2_n10k_d3", 20000, 18000, 3, 0.002, 1e-6, 0),
    ("c2_n10k_d3", 20000, 18000, 3, 0.002, 1e-6, 1),
    ("c2_n10k_d3", 16000, 17000, 2, 0.0005, 1e-5, 0),
    # d = 4..8: records of 8 and 12 floats; clustered clouds, so that whole
    # cluster pairs are skipped
    ("clustered", 3000, 2600, 4, 0.003, 1e-4, 0),
    ("clustered", 3000, 2500, 5, 0.003, 1e-4, 1),
    ("clustered", 3000, 2600, 8, 0.003, 1e-5, 0),
    ("clustered", 2900, 2700, 7, 0.002, 1e-6, 1),
    # 36 x 32 blocks at d = 8: the two-level cull runs
    ("clustered", 4600, 4100, 8, 0.002, 1e-6, 0),
])
def test_screening_decisions_match_oracle(name, n, m, d, eps, tau, side):
    inp, f32, g32 = _screen_case(name, n, m, d, eps, 6)
    t = to_dev(dict(inp, f=f32, g=g32))
    counts, lists = fs.fs_sparse_screen(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], tau, side)
    counts, lists = counts.cpu().numpy(), lists.cpu().numpy()
    px, py = bsp.morton_order(inp["X"], inp["Y"])
    Xs, as_, Ys, bs = inp["X"][px], inp["a"][px], inp["Y"][py], inp["b"][py]
    cx, wx = bsp.block_stats(Xs, as_)
    cy, wy = bsp.block_stats(Ys, bs)
    U, sig = bsp.block_bounds(Xs, as_, f32.astype(np.float64)[px], Ys, bs,
                              g32.astype(np.float64)[py], eps, cx, cy)
    w_out = wx if side == 0 else wy
    if side == 1:
        U, sig = U.T, sig.T
    nO, nIn = U.shape
    T = np.log2(np.float64(tau)) + np.log2(w_out.astype(np.float64)) - np.log2(nIn)
    gap = U + sig - T[:, None]
    near_max = U >= U.max(axis=1, keepdims=True) - MARGIN
    gpu = np.zeros((nO, nIn), dtype=bool)
    for o in range(nO):
        row = lists[o, :counts[o]]
        assert counts[o] >= 1
        assert np.all(np.diff(row) > 0) and row.min() >= 0 and row.max() < nIn
        gpu[o, row] = True
    must_keep = gap >= MARGIN
    must_skip = (gap <= -MARGIN) & ~near_max
    assert np.all(gpu[must_keep]), "a block the bound keeps was skipped"
    assert not np.any(gpu[must_skip]), "a block the bound skips was kept"
    # the cases are chosen so that the screening is not trivial
    assert 0.0 < must_skip.mean() and gpu.mean() < 0.95


@pytest.mark.parametrize("n,m,d", [(1, 1, 1), (7, 300, 2), (130, 129, 3), (1000, 1300, 3),
                                   (2049, 700, 1), (1000, 1300, 4), (700, 900, 5), (129, 130, 6),
                                   (300, 257, 7), (513, 1100, 8)])
def test_without_screening_equals_dense_oracle(n, m, d):
    inp = random_cloud(n, m, d, seed=50 + n, weights="lognormal")
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.05, coarse_iters=0,
                                   max_iters=15, tau=0.0)
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], 0.05, 15)
    tol = F_TOL_FMA * C.max()
    assert max_abs(np64(f), fr) <= tol
    assert max_abs(np64(g), gr) <= tol
    assert rep["iters"] == 15
    assert rep["kept_pairs"] == rep["passes"] * n * m


@pytest.mark.parametrize("name,n,d,eps,tau", [("c2_n10k_d3", 2600, 1, 0.001, 1e-6),
                                              ("c2_n10k_d3", 3000, 2, 0.002, 1e-4),
                                              ("c1_n512_d2", 2200, 2, 0.02, 1e-5)])
def test_screened_solve_matches_oracle(name, n, d, eps, tau):
    inp = make_inputs(name, n=n, m=n - 300, d=d)
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], eps, coarse_iters=20,
                                   max_iters=25, tau=tau)
    fr, gr, orep = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 20, 25, tau)
    C = orc.cost(inp["X"], inp["Y"])
    tol = F_TOL_FMA * C.max()
    assert max_abs(np64(f), fr) <= tol
    assert max_abs(np64(g), gr) <= tol
    assert rep["iters"] == orep["iters"] == 25
    # work per pass within 2 % (borderline blocks may differ)
    per_gpu = rep["kept_pairs"] / rep["passes"]
    per_orc = orep["kept_pairs"] / orep["halves"]
    assert abs(per_gpu / per_orc - 1.0) < 0.02
    assert per_gpu < 0.9 * n * (n - 300)
    assert rep["residual"] == pytest.approx(orep["residual"], rel=1e-2, abs=1e-5)


@pytest.mark.parametrize("online_iters,eps", [(0, 0.002), (-1, 0.002), (-1, 0.0005)])
def test_reference_offsets_with_fixups_match_oracle(online_iters, eps):
    """After `online_iters` iterations a row's exponent offset comes from its
    previous LSE, read from its bias slot (through the block's affine fit of
    those LSEs).  With -1 that holds from the first update of a cold start,
    where the offset implied by f = g = 0 is far below the row's LSE (checked
    on the oracle).  At eps = 0.0005 the gap passes 200 log2 units for about
    1 % of the rows, beyond the guarded range even for a row at the top of
    its block's fit, so those rows go through the fixup (counted in the
    report).  The potentials must match the oracle either way."""
    inp = make_inputs("c2_n10k_d3", n=2000, m=1900, d=2)
    tau = 1e-6
    C = orc.cost(inp["X"], inp["Y"])
    e = orc.as_eps(eps)
    if online_iters == -1:
        # offset from f = 0: log2 a_i - ((0 - |x~|^2) L/eps + log2 a_i) = |x~|^2 L/eps;
        # LSE2 of the first update: (|x~|^2 - f_1) L/eps; gap = -f_1 L/eps
        f1, _, _ = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 0, 1, tau)
        # (f_1 = -eps LSE over the kept blocks; the gap is independent of the centring)
        gap = -f1 / (e * np.log(2.0))
        assert gap.min() < -64
        if eps < 0.001:
            assert gap.min() < -200
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], eps, coarse_iters=0,
                                   max_iters=8, tau=tau, online_iters=online_iters)
    fr, gr, _ = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 0, 8, tau)
    tol = F_TOL_FMA * C.max()
    assert max_abs(np64(f), fr) <= tol
    assert max_abs(np64(g), gr) <= tol
    if online_iters == -1 and eps < 0.001:
        assert rep["fixed_rows"] > 0
    if online_iters == 0:
        # settled offsets: a fixup is the exception
        assert rep["fixed_rows"] <= 0.01 * rep["passes"] * 2000


@pytest.mark.parametrize("n,m,d,eps,tau", [(2000, 1900, 4, 0.002, 1e-6), (2200, 2000, 5, 0.003, 1e-5),
                                           (2600, 2300, 8, 0.003, 1e-5)])
def test_screened_solve_above_three_dimensions_matches_oracle(n, m, d, eps, tau):
    """d = 4..8 (records of 8 and 12 floats, the kept blocks staged in 64- and
    32-column chunks) on clustered clouds: the coarse stage, the screenings
    and the reference-offset updates after two online iterations."""
    inp = clustered_cloud(n, m, d, 12 if d > 4 else 10, 0.03 if d > 4 else 0.04, seed=400 + d)
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], eps, coarse_iters=20,
                                   max_iters=25, tau=tau)
    fr, gr, orep = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 20, 25, tau)
    C = orc.cost(inp["X"], inp["Y"])
    tol = F_TOL_FMA * C.max()
    assert max_abs(np64(f), fr) <= tol
    assert max_abs(np64(g), gr) <= tol
    per_gpu = rep["kept_pairs"] / rep["passes"]
    per_orc = orep["kept_pairs"] / orep["halves"]
    assert abs(per_gpu / per_orc - 1.0) < 0.02
    assert per_gpu < 0.9 * n * m
    assert rep["residual"] == pytest.approx(orep["residual"], rel=1e-2, abs=1e-5)


@pytest.mark.parametrize("d,eps", [(8, 0.003), (8, 0.00004), (5, 0.00004)])
def test_reference_offsets_above_three_dimensions_match_oracle(d, eps):
    """Reference offsets from the first update (online_iters = -1) at d = 5
    and 8: the block's affine fit of the previous LSEs has 5 or 8 slopes.  At
    eps = 4e-5 the cold-start gap passes 200 log2 units (checked on the
    oracle), so rows go through the fixup at D = 8."""
    inp = clustered_cloud(2000, 1800, d, 12, 0.03, seed=500 + d)
    tau = 1e-6
    if eps < 0.001:
        f1, _, _ = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 0, 1, tau)
        gap = -f1 / (orc.as_eps(eps) * np.log(2.0))
        assert gap.min() < -200
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], eps, coarse_iters=0,
                                   max_iters=8, tau=tau, online_iters=-1)
    fr, gr, _ = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 0, 8, tau)
    C = orc.cost(inp["X"], inp["Y"])
    tol = F_TOL_FMA * C.max()
    assert max_abs(np64(f), fr) <= tol
    assert max_abs(np64(g), gr) <= tol
    if eps < 0.001:
        assert rep["fixed_rows"] > 0


def test_reference_offsets_with_many_fixups_match_oracle():
    """A cold start with reference offsets (online_iters = -1) at eps = 5e-5:
    more than 2000 of the 8000 rows start over 250 log2 units from their LSE
    (checked on the oracle), so the first update lists more than 1216 rows
    and the fixup runs one CTA per row instead of a cluster per row."""
    eps, tau = 5e-5, 1e-6
    inp = make_inputs("c2_n10k_d3", n=8000, m=7600, d=2)
    f1, _, _ = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 0, 1, tau)
    gap = -f1 / (orc.as_eps(eps) * np.log(2.0))
    assert (gap < -250).sum() > 2000
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], eps, coarse_iters=0,
                                   max_iters=4, tau=tau, online_iters=-1)
    fr, gr, _ = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 0, 4, tau)
    C = orc.cost(inp["X"], inp["Y"])
    assert max_abs(np64(f), fr) <= F_TOL_FMA * C.max()
    assert max_abs(np64(g), gr) <= F_TOL_FMA * C.max()
    assert rep["fixed_rows"] > 1216


def test_screened_solve_with_lognormal_weights_matches_oracle():
    """Non-uniform weights: block weights, and with them the per-block
    thresholds, vary across the blocks."""
    inp = random_cloud(2600, 2300, 2, seed=77, spread=0.3, weights="lognormal")
    eps, tau = 0.003, 1e-5
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], eps, coarse_iters=15,
                                   max_iters=20, tau=tau)
    fr, gr, orep = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 15, 20, tau)
    C = orc.cost(inp["X"], inp["Y"])
    assert max_abs(np64(f), fr) <= F_TOL_FMA * C.max()
    assert max_abs(np64(g), gr) <= F_TOL_FMA * C.max()
    assert rep["kept_pairs"] < 0.9 * rep["passes"] * 2600 * 2300


def test_degenerate_clouds():
    """Every point of X at one place and every point of Y at another: the
    bounding box has zero extent on every axis (all Morton codes equal, the
    order is the identity) and the blocks have zero extents."""
    X = np.tile(np.array([[0.25, -0.5, 1.0]], np.float32), (300, 1))
    Y = np.tile(np.array([[0.75, 0.5, 0.0]], np.float32), (200, 1))
    inp = dict(X=X, Y=Y, a=np.full(300, 1 / 300, np.float32), b=np.full(200, 1 / 200, np.float32))
    t = to_dev(inp)
    px, py = fs.fs_morton_order(t["X"], t["Y"])
    np.testing.assert_array_equal(px.cpu().numpy(), np.arange(300))
    np.testing.assert_array_equal(py.cpu().numpy(), np.arange(200))
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.05, coarse_iters=3,
                                   max_iters=4, tau=1e-6)
    fr, gr, _ = bsp.solve(X, inp["a"], Y, inp["b"], 0.05, 3, 4, 1e-6)
    C = orc.cost(X, Y)
    assert max_abs(np64(f), fr) <= F_TOL_FMA * C.max()
    assert max_abs(np64(g), gr) <= F_TOL_FMA * C.max()


def test_coarse_stage_alone_matches_oracle():
    inp = make_inputs("c2_n10k_d3", n=3000, m=2700)
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.01, coarse_iters=40,
                                   max_iters=0, tau=1e-6)
    px, py = bsp.morton_order(inp["X"], inp["Y"])
    fs_, gs_, (cx, wx, cy, wy), _ = bsp.coarse_potentials(inp["X"][px], inp["a"][px],
                                                          inp["Y"][py], inp["b"][py], 0.01, 40)
    fr = np.empty(3000)
    gr = np.empty(2700)
    fr[px], gr[py] = fs_, gs_
    Cc = orc.cost(cx, cy)
    assert max_abs(np64(f), fr) <= F_TOL_FMA * Cc.max()
    assert max_abs(np64(g), gr) <= F_TOL_FMA * Cc.max()
    assert rep["iters"] == 0


@pytest.mark.parametrize("tol,rounds,checks", [(0.0, 2, 3), (1e12, 4, 1)])
def test_lift_check_matches_oracle(tol, rounds, checks):
    """The lift check: lift_samples points evenly spaced in Morton order, the
    mean relative row-marginal error of the dense plan at the lifted
    potentials; a zero tolerance runs every extra centroid round, a loose one
    passes at once.  Rounds, error and the potentials after the fine
    iterations against the oracle."""
    inp = make_inputs("c2_n10k_d3", n=1500, m=1300)
    t = to_dev(inp)
    kw = dict(coarse_iters=5, max_iters=3, tau=1e-6, lift_samples=200, lift_tol=tol,
              lift_rounds=rounds)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.01, **kw)
    fr, gr, orep = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.01, 5, 3, 1e-6,
                             lift_samples=200, lift_tol=tol, lift_rounds=rounds)
    assert rep["lift_checks"] == orep["lift_checks"] == checks
    assert rep["lift_error"] == pytest.approx(orep["lift_error"], rel=1e-2)
    C = orc.cost(inp["X"], inp["Y"])
    assert max_abs(np64(f), fr) <= F_TOL_FMA * C.max()
    assert max_abs(np64(g), gr) <= F_TOL_FMA * C.max()
    if checks == 1:
        # a check that passes changes nothing
        f0, g0, rep0 = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.01, coarse_iters=5,
                                          max_iters=3, tau=1e-6)
        assert rep0["lift_checks"] == 0 and rep0["lift_error"] == -1.0
        np.testing.assert_array_equal(f.cpu().numpy(), f0.cpu().numpy())


def test_stopping_rule_matches_oracle():
    inp = make_inputs("c2_n10k_d3", n=1500, m=1500, d=2)
    t = to_dev(inp)
    kw = dict(coarse_iters=30, max_iters=300, tau=1e-5, target=5e-3, check_every=5)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.01, **kw)
    fr, gr, orep = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.01, 30, 300, 1e-5,
                             target=5e-3, check_every=5)
    assert rep["residual"] <= 5e-3 and orep["residual"] <= 5e-3
    assert rep["iters"] % 5 == 0 and abs(rep["iters"] - orep["iters"]) <= 5
    if rep["iters"] == orep["iters"]:
        C = orc.cost(inp["X"], inp["Y"])
        assert max_abs(np64(f), fr) <= F_TOL_FMA * C.max()


def test_host_buffers_give_the_same_potentials():
    inp = make_inputs("c2_n10k_d3", n=1500, m=1400)
    t = to_dev(inp)
    fd, gd, _ = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.01, coarse_iters=10,
                                   max_iters=10, tau=1e-6)
    fh, gh, _ = fs.fs_sparse_solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.01, coarse_iters=10,
                                   max_iters=10, tau=1e-6)
    np.testing.assert_array_equal(fd.cpu().numpy(), fh)
    np.testing.assert_array_equal(gd.cpu().numpy(), gh)


def test_warm_start_continues_the_iteration():
    """coarse_iters = 0 starts from the caller's (f, g): 10 + 10 iterations
    equal 20 (up to the float32 rounding of the handed-over potentials)."""
    inp = make_inputs("c2_n10k_d3", n=2000, m=1800)
    t = to_dev(inp)
    f1, g1, _ = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.01, coarse_iters=10,
                                   max_iters=20, tau=0.0)
    f2, g2, _ = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.01, coarse_iters=10,
                                   max_iters=10, tau=0.0)
    f3, g3, _ = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], 0.01, coarse_iters=0,
                                   max_iters=10, tau=0.0, f=f2, g=g2)
    C = orc.cost(inp["X"], inp["Y"])
    assert max_abs(np64(f3), np64(f1)) <= 1e-5 * C.max()
    assert max_abs(np64(g3), np64(g1)) <= 1e-5 * C.max()


def test_invalid_arguments_are_rejected():
    inp = to_dev(random_cloud(10, 10, 9, seed=1))
    with pytest.raises(fs.FlashSinkhornError) as e:
        fs.fs_sparse_solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.1)
    assert e.value.status == fs.FS_ERR_UNSUPPORTED
    inp = to_dev(random_cloud(10, 10, 2, seed=1))
    for kw in (dict(tau=1.0), dict(tau=-1e-3), dict(max_iters=-1), dict(target=-1.0),
               dict(lift_samples=10, coarse_iters=0), dict(lift_samples=10, coarse_iters=2,
                                                           lift_tol=-1.0),
               dict(lift_samples=-1, coarse_iters=2)):
        with pytest.raises(fs.FlashSinkhornError) as e:
            fs.fs_sparse_solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.1, **kw)
        assert e.value.status == fs.FS_ERR_INVALID_ARG


def test_screening_without_survivors_keeps_the_first_maximiser():
    """Output blocks whose potentials sit far below their marginals: every
    bound misses the threshold, so the list holds the first maximiser of U
    alone.  With 157 x 141 blocks the super-block cull runs and the rows are
    sized by its survivors (fewer entries than input blocks), so the maximiser
    is searched among the culled blocks without a whole-row scratch."""
    name, n, m, d, eps, tau = "c2_n10k_d3", 20000, 18000, 3, 0.002, 1e-6
    inp, f32, g32 = _screen_case(name, n, m, d, eps, 6)
    px, py = bsp.morton_order(inp["X"], inp["Y"])
    low = [3, 40, 77, 155]
    for o in low:
        f32[px[o * bsp.BLOCK:(o + 1) * bsp.BLOCK]] -= np.float32(400 * eps)
    t = to_dev(dict(inp, f=f32, g=g32))
    counts, lists = fs.fs_sparse_screen(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], tau, 0)
    counts, lists = counts.cpu().numpy(), lists.cpu().numpy()
    Xs, as_, Ys, bs = inp["X"][px], inp["a"][px], inp["Y"][py], inp["b"][py]
    cx, wx = bsp.block_stats(Xs, as_)
    cy, wy = bsp.block_stats(Ys, bs)
    U, sig = bsp.block_bounds(Xs, as_, f32.astype(np.float64)[px], Ys, bs,
                              g32.astype(np.float64)[py], eps, cx, cy)
    T = np.log2(np.float64(tau)) + np.log2(wx.astype(np.float64)) - np.log2(U.shape[1])
    for o in low:
        assert np.all(U[o] + sig[o] < T[o] - MARGIN)   # nothing passes the threshold
        assert counts[o] == 1
        top2 = np.sort(U[o])[-2:]
        if top2[1] - top2[0] > MARGIN:
            assert lists[o, 0] == int(np.argmax(U[o]))
    others = np.setdiff1d(np.arange(U.shape[0]), low)
    assert np.all(counts[others] >= 1)


def test_beyond_2_30_block_pairs_column_marginals():
    """n = m = 1.6e7 (125,000^2 > 2^30 block pairs): the kept lists live in a
    buffer sized at each screening from the super-block cull's survivors.
    The workload in its launch configuration; at the returned potentials the
    dense column marginals on sampled columns lie in [b_j, b_j + tau W_J]."""
    w = WORKLOADS["bs_n16m_d3"]
    eps, iters = w.stages[0]
    tau = w.tau
    inp = make_inputs(w.name)
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], eps, coarse_iters=w.coarse_iters,
                                   max_iters=iters, tau=tau)
    assert rep["iters"] == iters
    assert rep["blocks_x"] * rep["blocks_y"] > 2 ** 30
    assert rep["kept_pairs"] < 0.01 * rep["passes"] * w.n * w.m
    f64, g64 = np64(f), np64(g)
    del t, f, g
    _, py = bsp.morton_order(inp["X"], inp["Y"])
    _, wy = bsp.block_stats(inp["Y"][py], inp["b"][py])
    block_of = np.empty(w.m, dtype=np.int64)
    block_of[py] = np.arange(w.m) // bsp.BLOCK
    cols = np.linspace(0, w.m - 1, 24).astype(np.int64)
    g_upd = orc.f_update_rows(inp["Y"], inp["X"], inp["a"], eps, f64, cols)
    c = inp["b"][cols].astype(np.float64) * np.exp((g64[cols] - g_upd) / orc.as_eps(eps))
    b = inp["b"][cols].astype(np.float64)
    # float32 rounding at eps = 1.42e-4: half an ulp of |g_j| <= 3 is 8.4e-4 of eps,
    # and the scores reach ~1.5e4 log2 units (~1e-3 each, averaging over the rows)
    assert np.all(c >= b * (1 - 3e-3))
    assert np.all(c <= b * (1 + 3e-3) + tau * wy[block_of[cols]])


def test_full_size_column_marginals_within_the_screening_bound():
    """The benchmark's block-sparse workload in its launch configuration
    (n = m = 10^6, d = 3, the workload's eps, centroid iterations, fine
    iterations and tau): at the returned potentials (after a g-update) every
    dense column marginal c_j lies in [b_j, b_j + tau W_J] up to float32
    rounding -- the kept blocks carry exactly b_j and the skipped ones at
    most tau W_J.  Checked on sampled columns with the oracle's dense
    single-row update, which sees every column pair, kept or not."""
    w = WORKLOADS["bs_n1m_d3"]
    eps, iters = w.stages[0]
    tau = w.tau
    n = w.n
    inp = make_inputs(w.name)
    t = to_dev(inp)
    f, g, rep = fs.fs_sparse_solve(t["X"], t["a"], t["Y"], t["b"], eps, coarse_iters=w.coarse_iters,
                                   max_iters=iters, tau=tau)
    assert rep["iters"] == iters
    assert rep["kept_pairs"] < 0.2 * rep["passes"] * n * w.m
    f64, g64 = np64(f), np64(g)
    px, py = bsp.morton_order(inp["X"], inp["Y"])
    _, wy = bsp.block_stats(inp["Y"][py], inp["b"][py])
    block_of = np.empty(w.m, dtype=np.int64)
    block_of[py] = np.arange(w.m) // bsp.BLOCK
    cols = np.linspace(0, w.m - 1, 48).astype(np.int64)
    # g-update of column j from f (roles swapped): c_j / b_j = exp((g_j - g_upd_j) / eps)
    g_upd = orc.f_update_rows(inp["Y"], inp["X"], inp["a"], eps, f64, cols)
    c = inp["b"][cols].astype(np.float64) * np.exp((g64[cols] - g_upd) / orc.as_eps(eps))
    b = inp["b"][cols].astype(np.float64)
    # float32 rounding of g (|g| <= 3, eps = 1e-3: < 1.2e-4 relative in c_j) and of the
    # scores (|kappa x~.y~| up to ~2e3 log2 units: ~2e-4) stay below 1e-3
    assert np.all(c >= b * (1 - 1e-3))
    assert np.all(c <= b * (1 + 1e-3) + tau * wy[block_of[cols]])
