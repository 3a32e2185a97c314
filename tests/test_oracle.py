"""Pins of the float64 oracle against facts that do not come from the oracle.

Source: "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU"
(gist.science technical summary).  Problem statement: entropic OT with
squared-Euclidean cost solved by Sinkhorn.  Method 1: the log-domain update
f_i = -eps LSE_j[(g_j - C_ij)/eps + log b_j] and Proposition 1.  Method 3:
plan application as a weighted mean (barycentric projection, gradient).

Each pin is chosen so that a plausible slip in the oracle (a dropped log
weight, a sign, a swapped index or operand, a wrong denominator) fails one of
them; ``test_pins_catch_planted_mistakes`` checks that claim on mutants.
"""
import itertools
import math

import numpy as np
import pytest
from scipy.optimize import linear_sum_assignment
from scipy.spatial.distance import cdist

import oracle as orc
from streaming_sinkhorn_solver_gb300.workloads import make_inputs, random_cloud


def _cloud(n, m, d, seed, weights="uniform", spread=1.0):
    return random_cloud(n, m, d, seed, spread=spread, weights=weights)


# --- cost ------------------------------------------------------------------

def test_cost_matches_scipy_cdist():
    c = _cloud(37, 23, 5, 1)
    C = orc.cost(c["X"], c["Y"])
    ref = cdist(c["X"].astype(np.float64), c["Y"].astype(np.float64), "sqeuclidean")
    np.testing.assert_allclose(C, ref, rtol=1e-13, atol=1e-13)


# --- closed forms of one update -------------------------------------------

def test_single_pair_closed_form():
    """n = m = 1, a = b = 1: f = C_11 after the f-update, then g = 0, and the
    iterates stay there."""
    X = np.array([[0.3, -1.2]], np.float32)
    Y = np.array([[1.1, 0.4]], np.float32)
    C = orc.cost(X, Y)
    one = np.ones(1, np.float32)
    f, g = orc.sinkhorn(C, one, one, 0.07, 1)
    assert f[0] == pytest.approx(C[0, 0], abs=1e-14)
    assert g[0] == pytest.approx(0.0, abs=1e-14)
    f, g = orc.sinkhorn(C, one, one, 0.07, 5)
    assert f[0] == pytest.approx(C[0, 0], abs=1e-14)
    assert g[0] == pytest.approx(0.0, abs=1e-14)


def test_one_column_closed_form():
    """m = 1: LSE over one term, so f_i = C_i1 - g_1 - eps log b_1 exactly.
    Pins the sign of g, of C and of the log-weight."""
    c = _cloud(9, 1, 3, 2)
    C = orc.cost(c["X"], c["Y"])
    b = np.array([0.37], np.float32)
    g = np.array([0.3])
    eps = 0.2
    e = orc.as_eps(eps)
    f = orc.f_update(C, b, eps, g)
    np.testing.assert_allclose(f, C[:, 0] - 0.3 - e * math.log(float(b[0])), rtol=0, atol=1e-13)


def test_one_row_closed_form_g_update():
    """n = 1: g_j = C_1j - f_1 - eps log a_1 exactly (the symmetric update)."""
    c = _cloud(1, 11, 2, 3)
    C = orc.cost(c["X"], c["Y"])
    a = np.array([0.61], np.float32)
    f = np.array([-0.45])
    eps = 0.05
    e = orc.as_eps(eps)
    g = orc.g_update(C, a, eps, f)
    np.testing.assert_allclose(g, C[0, :] + 0.45 - e * math.log(float(a[0])), rtol=0, atol=1e-13)


def test_two_points_softmin_limit():
    """Two columns, one far away: the f-update tends to the soft-min picking
    the near column, f -> C_near - g_near - eps log b_near."""
    X = np.array([[0.0]], np.float32)
    Y = np.array([[0.1], [5.0]], np.float32)
    C = orc.cost(X, Y)
    b = np.array([0.25, 0.75], np.float32)
    eps = 0.01
    f = orc.f_update(C, b, eps, np.zeros(2))
    e = orc.as_eps(eps)
    # the far term is exp(-(25-0.01)/0.01) relative: far below double precision
    assert f[0] == pytest.approx(C[0, 0] - e * math.log(0.25), abs=1e-12)


def test_symmetric_two_by_two_converged_plan():
    """X = Y = {0, 1} on the line, uniform weights: by symmetry the converged
    plan is P = [[p, q], [q, p]] with p + q = 1/2 and p/q = exp(c/eps), i.e.
    p = 1 / (2 (1 + exp(-c/eps))), c = 1."""
    X = np.array([[0.0], [1.0]], np.float32)
    w = np.full(2, 0.5, np.float32)
    C = orc.cost(X, X)
    eps = 0.5
    f, g = orc.sinkhorn(C, w, w, eps, 200)
    P = orc.apply_plan(C, w, w, eps, f, g, np.eye(2, dtype=np.float32))
    p = 1.0 / (2.0 * (1.0 + math.exp(-1.0 / orc.as_eps(eps))))
    np.testing.assert_allclose(P, [[p, 0.5 - p], [0.5 - p, p]], atol=1e-13)


# --- Proposition 1 ---------------------------------------------------------

@pytest.mark.parametrize("n,m,d,eps", [(17, 29, 2, 0.05), (40, 33, 8, 0.3), (25, 31, 64, 0.1)])
def test_proposition1_identity(n, m, d, eps):
    """The direct C-form update equals the biased-dot-product LSE form with
    Q = sqrt2 X, K = sqrt2 Y, g_hat = g - ||y||^2, delta = eps log b."""
    c = _cloud(n, m, d, 10 + d, weights="lognormal", spread=1.0 / math.sqrt(d))
    C = orc.cost(c["X"], c["Y"])
    rng = np.random.default_rng(4)
    g = 0.1 * rng.standard_normal(m)
    f_direct = orc.f_update(C, c["b"], eps, g)
    f_prop1 = orc.f_update_prop1(c["X"], c["Y"], c["b"], eps, g)
    np.testing.assert_allclose(f_prop1, f_direct, rtol=0, atol=1e-11 * C.max())


def test_rows_variants_match_full():
    c = _cloud(30, 41, 6, 5, weights="lognormal")
    C = orc.cost(c["X"], c["Y"])
    rng = np.random.default_rng(6)
    g = 0.2 * rng.standard_normal(41)
    rows = np.array([0, 7, 29, 13])
    f = orc.f_update(C, c["b"], 0.2, g)
    np.testing.assert_allclose(orc.f_update_rows(c["X"], c["Y"], c["b"], 0.2, g, rows), f[rows],
                               rtol=0, atol=1e-13)
    f2 = 0.1 * rng.standard_normal(30)
    V = rng.standard_normal((41, 3)).astype(np.float32)
    full = orc.apply_plan(C, c["a"], c["b"], 0.2, f2, g, V)
    part = orc.apply_plan_rows(c["X"], c["a"], c["Y"], c["b"], 0.2, f2, g, V, rows)
    np.testing.assert_allclose(part, full[rows], rtol=1e-13, atol=1e-15)


# --- marginals -------------------------------------------------------------

def test_marginals_exact_after_each_half():
    """Right after an f-update the plan's row sums are a; right after a
    g-update its column sums are b (to rounding)."""
    c = _cloud(45, 38, 3, 7, weights="lognormal")
    a, b = c["a"], c["b"]
    C = orc.cost(c["X"], c["Y"])
    eps = 0.05
    g_old = np.zeros(38)
    f, g = None, g_old
    for _ in range(3):
        g_old = g
        f = orc.f_update(C, b, eps, g_old)
        row, _ = orc.marginals(C, a, b, eps, f, g_old)
        np.testing.assert_allclose(row, a, rtol=1e-12)
        g = orc.g_update(C, a, eps, f)
        _, col = orc.marginals(C, a, b, eps, f, g)
        np.testing.assert_allclose(col, b, rtol=1e-12)


def test_marginal_residuals_vanish_at_convergence():
    """Exactly balanced masses (32 uniform weights of 1/32): both residuals go
    to rounding level.  Weights cast to float32 carry a mass gap
    |sum a - sum b| of order 1e-8; then the residuals settle at that gap."""
    c = _cloud(32, 32, 2, 8)
    C = orc.cost(c["X"], c["Y"])
    eps = 0.2 * C.max()
    f, g = orc.sinkhorn(C, c["a"], c["b"], eps, 400)
    row, col = orc.marginals(C, c["a"], c["b"], eps, f, g)
    assert np.abs(row - c["a"]).sum() < 1e-13
    assert np.abs(col - c["b"]).sum() < 1e-13
    c = _cloud(30, 30, 2, 8, weights="lognormal")
    gap = abs(float(c["a"].astype(np.float64).sum() - c["b"].astype(np.float64).sum()))
    C = orc.cost(c["X"], c["Y"])
    f, g = orc.sinkhorn(C, c["a"], c["b"], eps, 400)
    row, col = orc.marginals(C, c["a"], c["b"], eps, f, g)
    assert np.abs(row - c["a"]).sum() < 2 * gap + 1e-13
    assert np.abs(col - c["b"]).sum() < 1e-13


def test_entropic_duality_links_dual_value_transport_cost_and_marginals():
    """For any potentials the plan's form gives log(P_ij / (a_i b_j)) =
    (f_i + g_j - C_ij)/eps, hence sum_ij P_ij log(P_ij / (a_i b_j)) =
    (<f, P1> + <g, P^T 1> - <P, C>)/eps.  At the Sinkhorn fixed point P1 = a
    and P^T 1 = b, and this is strong duality of entropic OT:
    <a, f> + <b, g> = <P, C> + eps KL(P | a x b).  The entropy term is
    evaluated here from the plan's definition on a scipy cost matrix, so
    the identity ties the oracle's marginals, transport cost and dual value
    to each other and to the plan."""
    c = _cloud(40, 35, 3, 12, weights="lognormal")
    a = c["a"].astype(np.float64)
    b = c["b"].astype(np.float64)
    Cs = cdist(c["X"].astype(np.float64), c["Y"].astype(np.float64), "sqeuclidean")
    C = orc.cost(c["X"], c["Y"])
    eps = orc.as_eps(0.3)

    def entropy_term(f, g):
        logr = (f[:, None] + g[None, :] - Cs) / eps        # log(P / (a x b))
        P = a[:, None] * b[None, :] * np.exp(logr)
        return float((P * logr).sum())

    # any potentials: the identity with the realised marginals
    f, g = orc.sinkhorn(C, c["a"], c["b"], eps, 3)
    g = g + 0.05                                           # off the last g-update
    row, col = orc.marginals(C, c["a"], c["b"], eps, f, g)
    tc = orc.transport_cost(C, c["a"], c["b"], eps, f, g)
    lhs = float(f @ row + g @ col)
    assert abs(lhs - (tc + eps * entropy_term(f, g))) <= 1e-12 * max(1.0, abs(lhs))
    # the fixed point: strong duality with the dual value
    f, g = orc.sinkhorn(C, c["a"], c["b"], eps, 500)
    tc = orc.transport_cost(C, c["a"], c["b"], eps, f, g)
    gap = abs(float(a.sum() - b.sum()))                    # float32 weights: masses differ slightly
    dual = orc.dual(c["a"], c["b"], f, g)
    scale = float(np.abs(f).max() + np.abs(g).max())
    assert abs(dual - (tc + eps * entropy_term(f, g))) <= 1e-10 + 4 * gap * scale


# --- invariances ------------------------------------------------------------

def test_gauge_invariance_of_plan_and_update_equivariance():
    c = _cloud(21, 19, 4, 9)
    C = orc.cost(c["X"], c["Y"])
    eps = 0.1
    rng = np.random.default_rng(10)
    g = 0.3 * rng.standard_normal(19)
    f = orc.f_update(C, c["b"], eps, g)
    V = rng.standard_normal((19, 2)).astype(np.float32)
    shift = 0.731
    P1 = orc.apply_plan(C, c["a"], c["b"], eps, f, g, V)
    P2 = orc.apply_plan(C, c["a"], c["b"], eps, f + shift, g - shift, V)
    np.testing.assert_allclose(P1, P2, rtol=1e-12, atol=1e-15)
    # f-update(g + s) = f-update(g) - s
    np.testing.assert_allclose(orc.f_update(C, c["b"], eps, g + shift), f - shift, atol=1e-12)


def test_translation_invariance():
    c = _cloud(24, 27, 3, 11)
    t = np.array([0.5, -2.0, 1.0], np.float32)
    eps = 0.1
    C0 = orc.cost(c["X"], c["Y"])
    C1 = orc.cost(c["X"] + t, c["Y"] + t)
    f0, g0 = orc.sinkhorn(C0, c["a"], c["b"], eps, 20)
    f1, g1 = orc.sinkhorn(C1, c["a"], c["b"], eps, 20)
    # the shifted fp32 inputs round differently: agreement to float32 input precision
    np.testing.assert_allclose(f1, f0, atol=1e-5 * C0.max())
    np.testing.assert_allclose(g1, g0, atol=1e-5 * C0.max())


def test_symmetric_problem_f_minus_g_constant():
    c = _cloud(20, 20, 2, 12, weights="lognormal")
    X, a = c["X"], c["a"]
    C = orc.cost(X, X)
    eps = 0.3 * C.max()
    f, g = orc.sinkhorn(C, a, a, eps, 300)
    diff = f - g
    assert np.ptp(diff) < 1e-10


# --- limits -----------------------------------------------------------------

def test_large_eps_plan_is_product_measure():
    c = _cloud(16, 14, 3, 13, weights="lognormal")
    C = orc.cost(c["X"], c["Y"])
    eps = 1e6 * C.max()
    f, g = orc.sinkhorn(C, c["a"], c["b"], eps, 3)
    V = np.random.default_rng(14).standard_normal((14, 2)).astype(np.float32)
    out = orc.apply_plan(C, c["a"], c["b"], eps, f, g, V)
    ref = c["a"].astype(np.float64)[:, None] * (c["b"].astype(np.float64) @ V.astype(np.float64))[None, :]
    np.testing.assert_allclose(out, ref, rtol=1e-5, atol=1e-9)


def _brute_force_ot(C):
    n = C.shape[0]
    best = min(sum(C[i, p[i]] for i in range(n)) for p in itertools.permutations(range(n)))
    return best / n


@pytest.mark.parametrize("n,seed", [(5, 21), (7, 22)])
def test_small_eps_cost_tends_to_exact_ot(n, seed):
    """Uniform weights, n = m <= 7: <P, C> -> exact OT found over all
    permutations, with 0 <= <P,C> - OT <= eps log n (the entropic problem
    adds eps KL(P | a x b), which is log n for a permutation plan)."""
    c = _cloud(n, n, 2, seed)
    C = orc.cost(c["X"], c["Y"])
    ot = _brute_force_ot(C)
    a, b = c["a"], c["b"]
    f = np.zeros(n)
    g = np.zeros(n)
    gaps = []
    for eps_rel in [1e-1, 3e-2, 1e-2, 3e-3, 1e-3]:
        eps = eps_rel * C.max()
        for _ in range(200):
            f, g = orc.sinkhorn(C, a, b, eps, 50, f, g)
            row, col = orc.marginals(C, a, b, eps, f, g)
            if np.abs(row - a).sum() + np.abs(col - b).sum() < 1e-9:
                break
        val = orc.transport_cost(C, a, b, eps, f, g)
        gap = val - ot
        e = orc.as_eps(eps)
        assert -1e-7 * C.max() <= gap <= e * math.log(n) + 1e-7 * C.max()
        gaps.append(gap)
    assert gaps[-1] < gaps[0]
    assert gaps[-1] < 2e-3 * C.max()


def test_small_eps_matches_linear_sum_assignment():
    """Larger uniform case: exact OT from scipy's assignment solver."""
    n = 40
    c = _cloud(n, n, 3, 23)
    C = orc.cost(c["X"], c["Y"])
    r, cidx = linear_sum_assignment(C)
    ot = C[r, cidx].sum() / n
    a, b = c["a"], c["b"]
    f = np.zeros(n)
    g = np.zeros(n)
    for eps_rel in [1e-1, 1e-2, 2e-3]:
        eps = eps_rel * C.max()
        f, g = orc.sinkhorn(C, a, b, eps, 3000, f, g)
    val = orc.transport_cost(C, a, b, eps, f, g)
    assert 0 <= val - ot + 1e-6 <= orc.as_eps(eps) * math.log(n) + 2e-6


# --- plan application and gradient -------------------------------------------

def test_barycentric_of_identity_coupling_limit():
    """Y a permutation of X, uniform weights, small eps: the plan approaches
    the permutation, so the barycentric projection maps x_i to its partner."""
    rng = np.random.default_rng(30)
    X = np.array([[0.25 * i, 0.25 * j] for i in range(3) for j in range(4)], np.float32)
    perm = rng.permutation(12)
    Y = X[perm] + np.float32(0.001)
    w = np.full(12, 1 / 12, np.float32)
    C = orc.cost(X, Y)
    eps = 1e-3 * C.max()
    f, g = orc.sinkhorn(C, w, w, 10 * eps, 500)
    f, g = orc.sinkhorn(C, w, w, eps, 2000, f, g)
    T = orc.barycentric(C, w, w, eps, f, g, Y)
    inv = np.argsort(perm)
    np.testing.assert_allclose(T, Y[inv], atol=1e-3)


def _dual_value(X, a, Y, b, eps, iters):
    C = orc.cost(X, Y)
    f, g = orc.sinkhorn(C, a, b, eps, iters)
    return orc.dual(a, b, f, g), C, f, g


def test_grad_x_matches_finite_differences():
    """At convergence, d/dx_i (<a,f*> + <b,g*>) = 2 (a_i x_i - (P Y)_i)
    (envelope theorem on the entropic dual)."""
    c = _cloud(8, 10, 3, 31, weights="lognormal")
    X, Y, a, b = c["X"], c["Y"], c["a"], c["b"]
    eps = 0.4
    iters = 400
    _, C, f, g = _dual_value(X, a, Y, b, eps, iters)
    grad = orc.grad_x(C, X, a, b, eps, f, g, Y)
    fd = np.zeros_like(grad)
    for i in range(X.shape[0]):
        for k in range(X.shape[1]):
            Xp = X.copy(); Xm = X.copy()
            Xp[i, k] = np.float32(X[i, k] + np.float32(2e-3))
            Xm[i, k] = np.float32(X[i, k] - np.float32(2e-3))
            h = float(Xp[i, k]) - float(Xm[i, k])
            fd[i, k] = (_dual_value(Xp, a, Y, b, eps, iters)[0]
                        - _dual_value(Xm, a, Y, b, eps, iters)[0]) / h
    np.testing.assert_allclose(grad, fd, rtol=2e-4, atol=2e-5 * np.abs(grad).max())


def test_workload_inputs_have_recipe_shapes():
    for name, (n, m, d) in {"c1_n512_d2": (512, 512, 2), "c2_n10k_d3": (300, 200, 3),
                            "c3_n50k_d64": (100, 90, 64), "c4_n50k_d512": (20, 30, 512),
                            "c5_n20k_m30k_d1024": (10, 15, 1024)}.items():
        inp = make_inputs(name, n=n, m=m)
        assert inp["X"].shape == (n, d) and inp["Y"].shape == (m, d)
        assert inp["X"].dtype == np.float32 and inp["a"].dtype == np.float32
        assert abs(float(inp["a"].astype(np.float64).sum()) - 1) < 1e-6
        assert (inp["a"] > 0).all() and (inp["b"] > 0).all()
    c4 = make_inputs("c4_n50k_d512", n=20, m=30)
    np.testing.assert_allclose(np.linalg.norm(c4["X"], axis=1), 1, atol=1e-6)


# --- cosine cost (the pages' Discussion: cosine as squared-Euclidean on
# normalised points, C = 2 - 2 cos) ---------------------------------------

def test_cosine_cost_special_values():
    """Same direction 0, orthogonal 2, opposite 4, whatever the lengths; a zero
    row costs 1 against a nonzero point and 0 against another zero row."""
    X = np.array([[2.0, 0.0], [0.0, 0.0]], np.float32)
    Y = np.array([[5.0, 0.0], [0.0, 0.3], [-1.0, 0.0], [0.0, 0.0]], np.float32)
    C = orc.cost_cosine(X, Y)
    np.testing.assert_allclose(C, [[0.0, 2.0, 4.0, 1.0], [1.0, 1.0, 1.0, 0.0]], atol=1e-15)


def test_cosine_cost_equals_squared_euclidean_on_unit_rows():
    """On unit rows 2 - 2 cos(x, y) = |x - y|^2: the definition against the
    squared-Euclidean oracle cost (a different formula)."""
    rng = np.random.default_rng(5)
    X = rng.standard_normal((40, 7))
    Y = rng.standard_normal((30, 7))
    X = (X / np.linalg.norm(X, axis=1, keepdims=True)).astype(np.float32)
    Y = (Y / np.linalg.norm(Y, axis=1, keepdims=True)).astype(np.float32)
    np.testing.assert_allclose(orc.cost_cosine(X, Y), orc.cost(X, Y), atol=2e-7)


def test_cosine_cost_invariant_to_positive_row_scaling():
    rng = np.random.default_rng(6)
    X = rng.standard_normal((25, 5)).astype(np.float32)
    Y = rng.standard_normal((20, 5)).astype(np.float32)
    s = rng.uniform(0.1, 10.0, (25, 1)).astype(np.float32)
    t = rng.uniform(0.1, 10.0, (20, 1)).astype(np.float32)
    np.testing.assert_allclose(orc.cost_cosine(X * s, Y * t), orc.cost_cosine(X, Y), atol=1e-6)


def test_grad_x_cosine_matches_finite_differences():
    """At convergence under the cosine cost, d/dx_i (<a,f*> + <b,g*>) equals
    the chain rule through the normalisation (envelope theorem)."""
    c = _cloud(6, 7, 3, 37, weights="lognormal")
    X, Y, a, b = c["X"], c["Y"], c["a"], c["b"]
    eps, iters = 0.3, 600

    def dual_cos(Xv):
        C = orc.cost_cosine(Xv, Y)
        f, g = orc.sinkhorn(C, a, b, eps, iters)
        return orc.dual(a, b, f, g), C, f, g

    _, C, f, g = dual_cos(X)
    grad = orc.grad_x_cosine(C, X, a, b, eps, f, g, Y)
    fd = np.zeros_like(grad)
    for i in range(X.shape[0]):
        for k in range(X.shape[1]):
            Xp = X.copy(); Xm = X.copy()
            Xp[i, k] = np.float32(X[i, k] + np.float32(2e-3))
            Xm[i, k] = np.float32(X[i, k] - np.float32(2e-3))
            h = float(Xp[i, k]) - float(Xm[i, k])
            fd[i, k] = (dual_cos(Xp)[0] - dual_cos(Xm)[0]) / h
    np.testing.assert_allclose(grad, fd, rtol=2e-4, atol=2e-5 * np.abs(grad).max())
    # the gradient is orthogonal to x_i (a cosine cost cannot change along it)
    assert np.abs(np.sum(grad * X.astype(np.float64), axis=1)).max() <= 1e-12 * np.abs(grad).max() * 10


# --- Hessian-vector product of the converged OT value (derived here; the
# pages name a streaming HVP without a formula) ---------------------------

def test_hvp_single_pair_closed_form():
    """n = m = 1: F = |x - y|^2, so H = 2 I at any eps."""
    X = np.array([[0.3, -1.2, 0.5]], np.float32)
    Y = np.array([[1.0, 0.25, -0.5]], np.float32)
    a = b = np.ones(1, np.float32)
    C = orc.cost(X, Y)
    f, g = orc.sinkhorn(C, a, b, 0.7, 3)
    V = np.array([[0.2, 1.5, -0.4]])
    np.testing.assert_allclose(orc.hvp_x(C, X, a, b, 0.7, f, g, Y, V), 2.0 * V, atol=1e-12)


def test_hvp_matches_finite_differences_of_the_gradient():
    c = _cloud(6, 7, 2, 41, weights="lognormal")
    X, Y, a, b = c["X"], c["Y"], c["a"], c["b"]
    eps, iters = 0.5, 800
    V = np.random.default_rng(3).standard_normal(X.shape)

    def grad_at(Xv):
        C = orc.cost(Xv, Y)
        f, g = orc.sinkhorn(C, a, b, eps, iters)
        return orc.grad_x(C, Xv, a, b, eps, f, g, Y)

    C = orc.cost(X, Y)
    f, g = orc.sinkhorn(C, a, b, eps, iters)
    hv = orc.hvp_x(C, X, a, b, eps, f, g, Y, V)
    h = 1e-3
    Xp = (X.astype(np.float64) + h * V).astype(np.float32)
    Xm = (X.astype(np.float64) - h * V).astype(np.float32)
    # the float32 rounding of X +- hV is part of the step actually taken
    dX = Xp.astype(np.float64) - Xm.astype(np.float64)
    fd = (grad_at(Xp) - grad_at(Xm)) / (2 * h)
    hv_taken = orc.hvp_x(C, X, a, b, eps, f, g, Y, dX / (2 * h))
    np.testing.assert_allclose(hv_taken, fd, rtol=1e-3, atol=1e-4 * np.abs(fd).max())
    assert np.abs(hv - hv_taken).max() <= 1e-2 * np.abs(hv).max()


def test_hvp_is_symmetric():
    """<U, H V> = <V, H U>: a Hessian is symmetric.  Exactly so only at an exact
    fixed point, which needs equal masses: dyadic uniform weights (1/8, 1/16)
    sum to 1 exactly in float32."""
    c = _cloud(8, 16, 3, 43)
    X, Y, a, b = c["X"], c["Y"], c["a"], c["b"]
    assert float(a.astype(np.float64).sum()) == float(b.astype(np.float64).sum()) == 1.0
    eps = 0.3
    C = orc.cost(X, Y)
    f, g = orc.sinkhorn(C, a, b, eps, 2000)
    rng = np.random.default_rng(4)
    U = rng.standard_normal(X.shape)
    V = rng.standard_normal(X.shape)
    lhs = float(np.sum(U * orc.hvp_x(C, X, a, b, eps, f, g, Y, V)))
    rhs = float(np.sum(V * orc.hvp_x(C, X, a, b, eps, f, g, Y, U)))
    assert abs(lhs - rhs) <= 1e-8 * max(abs(lhs), 1.0)
