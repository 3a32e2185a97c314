"""GPU parity of the cosine cost (C = 2 - 2 cos) against the float64 oracle's
cosine cost, which is written from the definition (not from normalised
differences), on both paths: potentials, plan application, barycentric map
of the normalised points, and the gradient with respect to the raw X."""
import numpy as np
import pytest

import oracle as orc
from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import make_inputs, random_cloud
from tests.gpu_util import APPLY_TOL, F_TOL_FMA, F_TOL_TENSOR, max_abs, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


def _normalised(P):
    P = np.asarray(P, np.float64)
    nrm = np.linalg.norm(P, axis=1, keepdims=True)
    return np.where(nrm > 0, P / np.where(nrm > 0, nrm, 1.0), 0.0)


@pytest.mark.parametrize("n,m,d,tol", [(700, 900, 3, F_TOL_FMA), (900, 700, 8, F_TOL_FMA),
                                       (640, 520, 64, F_TOL_TENSOR), (300, 280, 300, F_TOL_TENSOR)])
def test_cosine_potentials_match_oracle(n, m, d, tol):
    inp = random_cloud(n, m, d, seed=400 + d, weights="lognormal")
    inp["X"][:, 0] += 0.7          # not centred: the norms differ from row to row
    inp["X"][3] = 0.0              # one zero row
    eps, iters = 0.05, 20
    t = to_dev(inp)
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, iters, cost="cosine")
    C = orc.cost_cosine(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, iters)
    assert max_abs(np64(f), fr) <= tol * C.max()
    assert max_abs(np64(g), gr) <= tol * C.max()


@pytest.mark.parametrize("d", [3, 64, 300])
def test_cosine_plan_operators_match_oracle(d):
    """d = 300: the barycentric map and the gradient (k = d > 128) go through
    the 256-column output blocks of the tensor plan application."""
    inp = random_cloud(600, 500, d, seed=450 + d, weights="lognormal")
    inp["X"] *= np.linspace(0.2, 3.0, 600, dtype=np.float32)[:, None]
    eps = 0.1
    C = orc.cost_cosine(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, 30)
    f32, g32 = fr.astype(np.float32), gr.astype(np.float32)
    V = np.random.default_rng(d).standard_normal((500, 6)).astype(np.float32)
    t = to_dev(dict(inp, f=f32, g=g32, V=V))
    out = fs.fs_apply_plan(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"],
                           cost="cosine")
    assert rel_l2(np64(out), orc.apply_plan(C, inp["a"], inp["b"], eps, f32, g32, V)) <= APPLY_TOL
    T = fs.fs_barycentric(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], cost="cosine")
    Yh = _normalised(inp["Y"]).astype(np.float32)
    Tr = orc.apply_plan(C, inp["a"], inp["b"], eps, f32, g32, Yh) / inp["a"][:, None].astype(np.float64)
    assert rel_l2(np64(T), Tr) <= APPLY_TOL
    G = fs.fs_grad_x(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], cost="cosine")
    Gr = orc.grad_x_cosine(C, inp["X"], inp["a"], inp["b"], eps, f32, g32, inp["Y"])
    assert rel_l2(np64(G), Gr) <= APPLY_TOL


def test_cosine_equals_squared_euclidean_on_unit_rows():
    """c4's inputs are unit rows: the cosine and squared-Euclidean solves agree."""
    inp = make_inputs("c4_n50k_d512", n=1500, m=1400)
    t = to_dev(inp)
    f1, g1 = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.05, 10)
    f2, g2 = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.05, 10, cost="cosine")
    assert max_abs(np64(f1), np64(f2)) <= F_TOL_TENSOR * 4.0
    assert max_abs(np64(g1), np64(g2)) <= F_TOL_TENSOR * 4.0
