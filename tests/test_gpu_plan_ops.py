"""GPU parity of the Y-side plan operators, the dual value and the marginal
residuals against the float64 oracle, on both paths.

P^T is the oracle's plan with the roles exchanged (cost C^T, weights and
potentials swapped); the operators must match within 1e-3 relative L2 like
every plan application.
"""
import numpy as np
import pytest

import oracle as orc
from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import random_cloud
from tests.gpu_util import APPLY_TOL, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


def _state(n, m, d, seed, eps, iters):
    inp = random_cloud(n, m, d, seed=seed, spread=1.0 / np.sqrt(max(d, 4)), weights="lognormal")
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, iters)
    f32, g32 = fr.astype(np.float32), gr.astype(np.float32)
    return inp, C, f32, g32


@pytest.mark.parametrize("n,m,d,k", [(700, 900, 3, 5), (640, 520, 64, 7), (300, 420, 200, 16)])
def test_apply_plan_transposed(n, m, d, k):
    eps = 0.1
    inp, C, f32, g32 = _state(n, m, d, 11 + d, eps, 5)
    U = np.random.default_rng(d).standard_normal((n, k)).astype(np.float32)
    t = to_dev(dict(inp, U=U, f=f32, g=g32))
    out = fs.fs_apply_plan_t(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["U"])
    assert tuple(out.shape) == (m, k)
    ref = orc.apply_plan(C.T, inp["b"], inp["a"], eps, g32, f32, U)
    assert rel_l2(np64(out), ref) <= APPLY_TOL


@pytest.mark.parametrize("n,m,d", [(800, 600, 2), (512, 700, 64)])
def test_barycentric_and_grad_y(n, m, d):
    eps = 0.05
    inp, C, f32, g32 = _state(n, m, d, 23 + d, eps, 30)
    t = to_dev(dict(inp, f=f32, g=g32))
    T = fs.fs_barycentric_y(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"])
    Tr = orc.barycentric(C.T, inp["b"], inp["a"], eps, g32, f32, inp["X"])
    assert rel_l2(np64(T), Tr) <= APPLY_TOL
    G = fs.fs_grad_y(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"])
    Gr = orc.grad_x(C.T, inp["Y"], inp["b"], inp["a"], eps, g32, f32, inp["X"])
    assert rel_l2(np64(G), Gr) <= APPLY_TOL


def test_dual_value_device_and_host():
    inp, C, f32, g32 = _state(3000, 2500, 3, 31, 0.1, 10)
    ref = orc.dual(inp["a"], inp["b"], f32.astype(np.float64), g32.astype(np.float64))
    t = to_dev(dict(inp, f=f32, g=g32))
    v_dev = fs.fs_dual_value(t["a"], t["b"], t["f"], t["g"])
    v_host = fs.fs_dual_value(inp["a"], inp["b"], f32, g32)
    # double sums of fp32 products: equal up to double rounding of the order
    assert abs(v_dev - ref) <= 1e-12 * max(1.0, abs(ref)) * 3000
    assert v_dev == v_host


@pytest.mark.parametrize("d,iters", [(3, 3), (3, 40), (64, 3)])
def test_marginal_residuals(d, iters):
    """A few iterations leave O(0.1) row residuals; after a g-update the column
    residual is only rounding.  Absolute agreement within the plan tolerance
    times the total mass."""
    eps = 0.1
    inp, C, f32, g32 = _state(900, 800, d, 41 + d + iters, eps, iters)
    row, col = orc.marginals(C, inp["a"], inp["b"], eps, f32, g32)
    ref_r = float(np.abs(row - inp["a"]).sum())
    ref_c = float(np.abs(col - inp["b"]).sum())
    t = to_dev(dict(inp, f=f32, g=g32))
    r, c = fs.fs_marginal_residuals(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"])
    mass = float(inp["a"].sum())
    assert abs(r - ref_r) <= APPLY_TOL * mass
    assert abs(c - ref_c) <= APPLY_TOL * mass
    if iters >= 40:
        assert r < 1e-3 * mass


@pytest.mark.parametrize("d,iters", [(3, 3), (3, 40), (64, 3)])
def test_marginals_element_wise(d, iters):
    """The marginals themselves: P1 (the plan application with V = 1) and
    P^T 1 (the transposed application with U = 1), row by row and column by
    column against the oracle's plan sums, each within 1e-3 relative (sums of
    positive plan entries); the residuals the library reports are the L1
    distances of those vectors to a and b, up to the rounding of the sums."""
    eps = 0.1
    n, m = 900, 800
    inp, C, f32, g32 = _state(n, m, d, 41 + d + iters, eps, iters)
    row, col = orc.marginals(C, inp["a"], inp["b"], eps, f32, g32)
    t = to_dev(dict(inp, f=f32, g=g32, V=np.ones((m, 1), np.float32),
                    U=np.ones((n, 1), np.float32)))
    P1 = np64(fs.fs_apply_plan(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"]))[:, 0]
    PT1 = np64(fs.fs_apply_plan_t(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["U"]))[:, 0]
    assert np.max(np.abs(P1 - row) / row) <= APPLY_TOL
    assert np.max(np.abs(PT1 - col) / col) <= APPLY_TOL
    r, c = fs.fs_marginal_residuals(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"])
    mass = float(inp["a"].sum())
    assert abs(r - float(np.abs(P1 - inp["a"]).sum())) <= 1e-5 * mass
    assert abs(c - float(np.abs(PT1 - inp["b"]).sum())) <= 1e-5 * mass
