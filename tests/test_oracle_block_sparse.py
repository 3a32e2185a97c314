"""Pins of the block-sparse oracle (``oracle/block_sparse.py``) against facts
that do not come from it.

Source: "FlashSinkhorn 2: Block-Sparse Entropic Optimal Transport" (patty.io
post): Morton ordering of the points, a coarse solve between cell centroids
whose potentials the points inherit, block screening by a bound on each
block's plan mass, and a per-row / per-column bound on what the skipped
tiles can change.

* Z-order: an independent recursive 2^d-tree traversal of integer grids.
* Quantisation: in one dimension the Morton order is the order of the
  coordinates.
* The block bound: never below the brute-force block mass; equal to it for
  blocks of one point.
* The screening: the brute-force omitted mass of every output block is
  below tau times its weight; tau = 0 keeps everything.
* The coarse stage: with one point per cell it is the dense oracle.
* The iteration: with tau = 0 it is the dense oracle's Sinkhorn; with
  tau > 0 it converges to the dense fixed point.
``test_pins_catch_planted_block_sparse_mistakes`` plants slips in a copy of
the oracle's source and checks that a pin fails for each.
"""
import sys
import types

import numpy as np
import pytest

import oracle as orc
import oracle.block_sparse as bsp
from streaming_sinkhorn_solver_gb300.workloads import make_inputs, random_cloud


# --- Morton order ------------------------------------------------------------

def _ztree_order(q: np.ndarray, bits: int) -> np.ndarray:
    """Z-order by recursion: split the cell into its 2^d children (child
    index sum_k [q_k in upper half] 2^k), visit the children in index order,
    keep the input order inside a leaf."""
    d = q.shape[1]

    def rec(idx, level):
        if level < 0 or len(idx) <= 1:
            return list(idx)
        out = []
        child = np.zeros(len(idx), dtype=np.int64)
        for k in range(d):
            child += ((q[idx, k] >> level) & 1) << k
        for c in range(2 ** d):
            out += rec(idx[child == c], level - 1)
        return out

    return np.array(rec(np.arange(len(q)), bits - 1), dtype=np.int64)


@pytest.mark.parametrize("d", [1, 2, 3])
def test_morton_order_is_recursive_ztree_order(d):
    """Points on the integer lattice of a 2^21 grid whose box is [0, 2^21]:
    the float32 quantisation is the identity (the corner point at 2^21 is
    clamped), so the code order must equal the recursive traversal."""
    rng = np.random.default_rng(10 + d)
    G = 2 ** 21
    pts = rng.integers(0, G, size=(300, d))
    pts[:40] = rng.integers(0, 4, size=(40, d))          # dense corner, many ties
    pts[40:60] = pts[100:120]                             # exact duplicates
    X = pts.astype(np.float32)
    Y = np.vstack([np.zeros((1, d)), np.full((1, d), G)]).astype(np.float32)
    lo, hi = bsp.morton_box(X, Y)
    assert np.all(lo == 0) and np.all(hi == G)
    order = np.argsort(bsp.morton_codes(X, lo, hi), kind="stable")
    q = np.clip(pts, 0, G - 1).astype(np.int64)
    np.testing.assert_array_equal(order, _ztree_order(q, 21))


@pytest.mark.parametrize("d,bits", [(4, 15), (5, 12), (8, 7)])
def test_morton_order_is_recursive_ztree_order_in_more_dimensions(d, bits):
    """The same pin for d = 4, 5 and 8, whose codes quantise each axis to
    2^floor(63 / d) cells (15, 12 and 7 bits) so that they fit 64 bits."""
    assert bsp.morton_bits(d) == bits
    rng = np.random.default_rng(20 + d)
    G = 2 ** bits
    pts = rng.integers(0, G, size=(400, d))
    pts[:50] = rng.integers(0, 2, size=(50, d))           # dense corner, many ties
    pts[50:70] = pts[200:220]                             # exact duplicates
    X = pts.astype(np.float32)
    Y = np.vstack([np.zeros((1, d)), np.full((1, d), G)]).astype(np.float32)
    lo, hi = bsp.morton_box(X, Y)
    order = np.argsort(bsp.morton_codes(X, lo, hi), kind="stable")
    q = np.clip(pts, 0, G - 1).astype(np.int64)
    np.testing.assert_array_equal(order, _ztree_order(q, bits))


def test_morton_codes_small_grid_by_hand():
    """The four cells of a 2 x 2 grid in two dimensions come in Z order
    (0,0), (1,0), (0,1), (1,1): codes 0, 1, 2, 3 at the top level."""
    G = float(2 ** 21)
    X = np.array([[0.75, 0.75], [0.25, 0.75], [0.75, 0.25], [0.25, 0.25]], np.float32) * G
    Y = np.array([[0.0, 0.0], [G, G]], np.float32)
    lo, hi = bsp.morton_box(X, Y)
    codes = bsp.morton_codes(X, lo, hi)
    top = codes >> np.uint64(40)              # the most significant 2-bit digit
    np.testing.assert_array_equal(top, [3, 2, 1, 0])


def test_morton_order_in_one_dimension_is_coordinate_order():
    rng = np.random.default_rng(3)
    x = rng.permutation(5000).astype(np.float32)[:, None] * np.float32(7.0)
    px, py = bsp.morton_order(x, x[:10])
    np.testing.assert_array_equal(px, np.argsort(x[:, 0], kind="stable"))


# --- block statistics and the coarse stage -------------------------------------

def test_block_stats_of_single_points_are_the_points():
    c = random_cloud(37, 5, 3, 4, weights="random")
    cx, wx = bsp.block_stats(c["X"], c["a"], block=1)
    np.testing.assert_array_equal(cx, c["X"])
    np.testing.assert_array_equal(wx, c["a"])


def test_block_stats_weighted_mean():
    c = random_cloud(300, 5, 2, 5, weights="random")
    cx, wx = bsp.block_stats(c["X"], c["a"], block=64)
    for I in range(len(cx)):
        sl = slice(64 * I, min(64 * I + 64, 300))
        np.testing.assert_allclose(cx[I], np.average(c["X"][sl].astype(np.float64), axis=0,
                                                     weights=c["a"][sl]), rtol=1e-6, atol=1e-7)
        assert wx[I] == pytest.approx(float(np.sum(c["a"][sl], dtype=np.float64)), rel=1e-7)


def test_coarse_stage_with_one_point_per_cell_is_the_dense_solve():
    c = random_cloud(40, 33, 2, 6, weights="random")
    f, g, _, _ = bsp.coarse_potentials(c["X"], c["a"], c["Y"], c["b"], 0.1, 15, block=1)
    fr, gr = orc.sinkhorn(orc.cost(c["X"], c["Y"]), c["a"], c["b"], 0.1, 15)
    np.testing.assert_allclose(f, fr, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g, gr, rtol=0, atol=1e-12)


# --- the lift check --------------------------------------------------------------

def test_lift_sample_positions_are_evenly_spaced_and_distinct():
    assert list(bsp.lift_sample(10, 4)) == [0, 2, 5, 7]
    assert list(bsp.lift_sample(3, 8)) == [0, 1, 2]
    r = bsp.lift_sample(1000, 64)
    assert len(np.unique(r)) == 64 and r.min() == 0 and r.max() < 1000


def test_lift_error_is_the_sampled_relative_row_marginal_error():
    """Against the dense oracle's plan marginals (P 1 summed from the plan
    entries), not the f-update identity the check uses."""
    c = random_cloud(300, 260, 3, 12, weights="random")
    C = orc.cost(c["X"], c["Y"])
    f, g = orc.sinkhorn(C, c["a"], c["b"], 0.1, 3)
    f = f + 0.01 * np.sin(np.arange(300))          # away from an f-update's exact rows
    rows = bsp.lift_sample(300, 37)
    r, _ = orc.marginals(C, c["a"], c["b"], 0.1, f, g)
    want = np.mean(np.abs(r[rows] / c["a"][rows].astype(np.float64) - 1.0))
    got = bsp.lift_error(c["X"], c["Y"], c["b"], 0.1, f, g, rows)
    assert got == pytest.approx(want, rel=1e-10)
    # after an f-update the rows are exact
    f1 = orc.f_update(C, c["b"], 0.1, g)
    assert bsp.lift_error(c["X"], c["Y"], c["b"], 0.1, f1, g, rows) < 1e-12


def test_coarse_stage_continues_like_one_longer_solve():
    """Two rounds of k centroid iterations, the second from where the first
    stopped, are 2k iterations from zero: the lift check's extra rounds."""
    inp = make_inputs("c2_n10k_d3", n=1500, m=1300)
    px, py = bsp.morton_order(inp["X"], inp["Y"])
    args = (inp["X"][px], inp["a"][px], inp["Y"][py], inp["b"][py], 0.01)
    _, _, _, (F1, G1) = bsp.coarse_potentials(*args, 7)
    f2, g2, _, _ = bsp.coarse_potentials(*args, 7, F0=F1, G0=G1)
    f14, g14, _, _ = bsp.coarse_potentials(*args, 14)
    np.testing.assert_allclose(f2, f14, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g2, g14, rtol=0, atol=1e-12)


def test_lift_check_rounds():
    """A loose tolerance passes the first check and changes nothing; a zero
    tolerance runs every extra round, which is the longer centroid solve."""
    inp = make_inputs("c2_n10k_d3", n=1500, m=1300)
    args = (inp["X"], inp["a"], inp["Y"], inp["b"], 0.01)
    f0, g0, r0 = bsp.solve(*args, 5, 3, 1e-6)
    f1, g1, r1 = bsp.solve(*args, 5, 3, 1e-6, lift_samples=200, lift_tol=1e9, lift_rounds=4)
    assert r1["lift_checks"] == 1 and r0["lift_checks"] == 0
    np.testing.assert_array_equal(f1, f0)
    f2, g2, r2 = bsp.solve(*args, 5, 3, 1e-6, lift_samples=200, lift_tol=0.0, lift_rounds=2)
    f3, g3, _ = bsp.solve(*args, 15, 3, 1e-6)
    assert r2["lift_checks"] == 3
    np.testing.assert_allclose(f2, f3, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g2, g3, rtol=0, atol=1e-12)
    assert r2["lift_error"] > 0.0


# --- the block bound and the screening -----------------------------------------

def _sorted_problem(name="c2_n10k_d3", n=900, m=700, eps=0.005, iters=8, block=32, d=None):
    inp = make_inputs(name, n=n, m=m, d=d)
    px, py = bsp.morton_order(inp["X"], inp["Y"])
    Xs, as_, Ys, bs = inp["X"][px], inp["a"][px], inp["Y"][py], inp["b"][py]
    C = orc.cost(Xs, Ys)
    fs, gs = orc.sinkhorn(C, as_, bs, eps, iters)
    cx, wx = bsp.block_stats(Xs, as_, block)
    cy, wy = bsp.block_stats(Ys, bs, block)
    return dict(Xs=Xs, as_=as_, Ys=Ys, bs=bs, C=C, fs=fs, gs=gs, cx=cx, wx=wx, cy=cy, wy=wy,
                eps=eps, block=block)


def _true_block_mass(p):
    e = orc.as_eps(p["eps"])
    P = (p["as_"].astype(np.float64)[:, None] * p["bs"].astype(np.float64)[None, :]
         * np.exp((p["fs"][:, None] + p["gs"][None, :] - p["C"]) / e))
    bi = bsp.block_ids(len(p["Xs"]), p["block"])
    bj = bsp.block_ids(len(p["Ys"]), p["block"])
    M = np.zeros((bi[-1] + 1, bj[-1] + 1))
    np.add.at(M, (bi[:, None], bj[None, :]), P)
    return M


@pytest.mark.parametrize("eps,d", [(0.05, None), (0.005, None), (0.02, 6), (0.05, 8)])
def test_block_bound_is_never_below_the_block_mass(eps, d):
    p = _sorted_problem(eps=eps, d=d)
    U, sig = bsp.block_bounds(p["Xs"], p["as_"], p["fs"], p["Ys"], p["bs"], p["gs"], eps,
                              p["cx"], p["cy"], p["block"])
    M = _true_block_mass(p)
    assert np.all(np.log2(np.maximum(M, 1e-300)) <= U + 1e-9)
    # Termwise, the bound drops only -|u_i - v_j|^2 from the exponent, so it
    # exceeds the mass by at most (r_I + r_J)^2 L/eps bits (r: block radii).
    def radii(P, c, B):
        r = np.linalg.norm(P.astype(np.float64) - c.astype(np.float64)[bsp.block_ids(len(P), B)], axis=1)
        return np.maximum.reduceat(r, np.arange(len(c)) * B)
    rx, ry = radii(p["Xs"], p["cx"], p["block"]), radii(p["Ys"], p["cy"], p["block"])
    slack = (rx[:, None] + ry[None, :]) ** 2 * bsp.L2E / orc.as_eps(eps)
    live = M > 1e-250
    assert np.all(U[live] <= np.log2(M[live]) + slack[live] + 1e-9)


def test_block_bound_of_single_points_is_the_plan_entry():
    c = random_cloud(23, 19, 3, 7, weights="random")
    C = orc.cost(c["X"], c["Y"])
    f, g = orc.sinkhorn(C, c["a"], c["b"], 0.2, 4)
    U, _ = bsp.block_bounds(c["X"], c["a"], f, c["Y"], c["b"], g, 0.2, c["X"], c["Y"], 1)
    e = orc.as_eps(0.2)
    logP = (np.log2(c["a"].astype(np.float64))[:, None] + np.log2(c["b"].astype(np.float64))[None, :]
            + (f[:, None] + g[None, :] - C) / e * bsp.L2E)
    np.testing.assert_allclose(U, logP, rtol=0, atol=1e-9)


@pytest.mark.parametrize("tau", [1e-2, 1e-4])
def test_screening_bounds_the_omitted_mass_per_block(tau):
    p = _sorted_problem(eps=0.002, n=1200, m=1000)
    U, sig = bsp.block_bounds(p["Xs"], p["as_"], p["fs"], p["Ys"], p["bs"], p["gs"], p["eps"],
                              p["cx"], p["cy"], p["block"])
    M = _true_block_mass(p)
    kx = bsp.screen(U, sig, p["wx"], tau, "x")
    ky = bsp.screen(U, sig, p["wy"], tau, "y")
    assert kx.mean() < 0.9 and ky.mean() < 0.9       # the screening skips something
    assert np.all(np.where(kx, 0, M).sum(axis=1) <= tau * p["wx"])
    assert np.all(np.where(ky, 0, M.T).sum(axis=1) <= tau * p["wy"])
    assert np.all(kx[np.arange(len(kx)), np.argmax(U, axis=1)])
    assert np.all(ky[np.arange(len(ky)), np.argmax(U.T, axis=1)])
    assert bsp.screen(U, sig, p["wx"], 0.0, "x").all()


# --- the block-sparse iteration --------------------------------------------------

@pytest.mark.parametrize("d", [3, 5, 8])
def test_iteration_without_screening_is_the_dense_solve(d):
    inp = make_inputs("c2_n10k_d3", n=600, m=500, d=d)
    f, g, rep = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.01, 0, 7, 0.0, block=64)
    fr, gr = orc.sinkhorn(orc.cost(inp["X"], inp["Y"]), inp["a"], inp["b"], 0.01, 7)
    cmax = orc.cost(inp["X"], inp["Y"]).max()
    np.testing.assert_allclose(f, fr, rtol=0, atol=1e-12 * cmax)
    np.testing.assert_allclose(g, gr, rtol=0, atol=1e-12 * cmax)
    assert rep["iters"] == 7 and rep["kept_pairs"] == 2 * 7 * 600 * 500


def test_masked_updates_make_the_kept_marginals_exact():
    """Right after a block-sparse f-update the row sums of the plan restricted
    to the kept blocks are a; right after the g-update the column sums over
    its kept blocks are b."""
    p = _sorted_problem(eps=0.003, n=700, m=600)
    e = orc.as_eps(p["eps"])
    bi = bsp.block_ids(700, p["block"])
    bj = bsp.block_ids(600, p["block"])

    def plan(f, g):
        return (p["as_"].astype(np.float64)[:, None] * p["bs"].astype(np.float64)[None, :]
                * np.exp((f[:, None] + g[None, :] - p["C"]) / e))

    U, sig = bsp.block_bounds(p["Xs"], p["as_"], p["fs"], p["Ys"], p["bs"], p["gs"], p["eps"],
                              p["cx"], p["cy"], p["block"])
    kx = bsp.screen(U, sig, p["wx"], 1e-3, "x")
    assert not kx.all()
    f = bsp.sparse_f_update(p["C"], p["bs"], p["eps"], p["gs"], kx, p["block"])
    rows = np.where(kx[bi][:, bj], plan(f, p["gs"]), 0.0).sum(axis=1)
    np.testing.assert_allclose(rows, p["as_"], rtol=1e-10)
    U, sig = bsp.block_bounds(p["Xs"], p["as_"], f, p["Ys"], p["bs"], p["gs"], p["eps"],
                              p["cx"], p["cy"], p["block"])
    ky = bsp.screen(U, sig, p["wy"], 1e-3, "y")
    assert not ky.all() and not np.array_equal(ky, kx.T)
    g = bsp.sparse_g_update(p["C"], p["as_"], p["eps"], f, ky, p["block"])
    cols = np.where(ky[bj][:, bi].T, plan(f, g), 0.0).sum(axis=0)
    np.testing.assert_allclose(cols, p["bs"], rtol=1e-10)


@pytest.mark.parametrize("d,eps,n,kept", [(2, 0.01, 800, 0.9), (5, 0.02, 1500, 0.97)])
def test_screened_iteration_converges_to_the_dense_fixed_point(d, eps, n, kept):
    """At the returned potentials the dense plan differs from the block-sparse
    one only by the omitted blocks, whose mass the screening bounds by tau in
    each marginal: |P_dense 1 - a|_1 <= residual + tau, |P_dense^T 1 - b|_1 <= tau."""
    inp = make_inputs("c2_n10k_d3", n=n, m=n, d=d)
    tau = 1e-4
    C = orc.cost(inp["X"], inp["Y"])
    f, g, rep = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, 30, 400, tau,
                          target=1e-5, check_every=10, block=32)
    assert rep["residual"] <= 1e-5 and rep["iters"] < 400
    # in five dimensions blocks of 32 uniform points are far from compact:
    # the screening still skips some
    assert rep["kept_pairs"] < kept * 2 * rep["iters"] * n * n
    r, c = orc.marginals(C, inp["a"], inp["b"], eps, f, g)
    assert np.abs(r - inp["a"]).sum() <= rep["residual"] + tau
    assert np.abs(c - inp["b"]).sum() <= tau


# --- planted mistakes -------------------------------------------------------------

MUTANTS = [
    ("interleave_as_concat", "codes |= bit << np.uint64(b * d + k)",
     "codes |= bit << np.uint64(k * bits + b)"),
    ("bound_linear_sign", "Z = psi[ri][:, None] - kap * (u @ D.T)",
     "Z = psi[ri][:, None] + kap * (u @ D.T)"),
    ("bound_no_linear_terms", "W = chi + kap * np.sum(v * D[bj], axis=1)", "W = chi + 0.0 * kap"),
    ("bound_dd_sign", "U[I] = A + B - dd", "U[I] = A + B + dd"),
    ("bound_no_logw", "+ np.log2(np.asarray(as_, np.float64))", ""),
    ("threshold_sign", "- np.log2(nIn)", "+ np.log2(nIn)"),
    ("stats_unweighted", "S[ok] = S[ok] + w[:, None] *", "S[ok] = S[ok] + 0 * w[:, None] + (1.0 / block) *"),
    ("sparse_g_reversed_row_blocks",
     "mask = keep_y[block_ids(C.shape[1], block)][:, block_ids(C.shape[0], block)]",
     "mask = keep_y[block_ids(C.shape[1], block)][:, block_ids(C.shape[0], block)[::-1]]"),
    ("screen_y_not_transposed", 'if side == "y":', "if False:"),
    ("lift_error_sign", "r = np.exp((np.asarray(fs, np.float64)[rows] - f_new) / as_eps(eps))",
     "r = np.exp((f_new - np.asarray(fs, np.float64)[rows]) / as_eps(eps))"),
    ("lift_restarts_from_zero", "F, G = sinkhorn(cost(cx, cy), wx, wy, eps, iters, F0, G0)",
     "F, G = sinkhorn(cost(cx, cy), wx, wy, eps, iters)"),
]

PINS = [
    lambda: test_morton_order_is_recursive_ztree_order(2),
    lambda: test_morton_codes_small_grid_by_hand(),
    lambda: test_block_stats_of_single_points_are_the_points(),
    lambda: test_block_stats_weighted_mean(),
    lambda: test_block_bound_is_never_below_the_block_mass(0.005, None),
    lambda: test_block_bound_of_single_points_is_the_plan_entry(),
    lambda: test_screening_bounds_the_omitted_mass_per_block(1e-2),
    lambda: test_masked_updates_make_the_kept_marginals_exact(),
    lambda: test_lift_error_is_the_sampled_relative_row_marginal_error(),
    lambda: test_coarse_stage_continues_like_one_longer_solve(),
]


def _load_mutant(old: str, new: str):
    src = open(bsp.__file__).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle._block_sparse_mutant")
    mod.__package__ = "oracle"
    mod.__file__ = bsp.__file__
    exec(compile(src.replace(old, new), bsp.__file__, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_block_sparse_mistakes(name, old, new, monkeypatch):
    mutant = _load_mutant(old, new)
    monkeypatch.setattr(sys.modules[__name__], "bsp", mutant)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake {name}"
