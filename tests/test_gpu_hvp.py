"""GPU Hessian-vector product against the dense float64 oracle (which solves
the differentiated fixed-point system by least squares), at converged
potentials.  The GPU solves the same system by conjugate gradients with plan
applications only."""
import numpy as np
import pytest

import oracle as orc
from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import make_inputs, random_cloud
from tests.gpu_util import APPLY_TOL, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


def _converged(n, m, d, seed, eps, iters=1500):
    inp = random_cloud(n, m, d, seed=seed, spread=1.0 / np.sqrt(max(d, 2)), weights="lognormal")
    C = orc.cost(inp["X"], inp["Y"])
    f, g = orc.sinkhorn(C, inp["a"], inp["b"], eps, iters)
    return inp, C, f.astype(np.float32), g.astype(np.float32)


@pytest.mark.parametrize("n,m,d,eps", [(300, 280, 2, 0.2), (260, 310, 3, 0.1), (200, 180, 8, 0.3)])
def test_hvp_fma_path_matches_oracle(n, m, d, eps):
    inp, C, f, g = _converged(n, m, d, 500 + d, eps)
    V = np.random.default_rng(d).standard_normal((n, d)).astype(np.float32)
    t = to_dev(dict(inp, f=f, g=g, V=V))
    hv = fs.fs_hvp_x(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"])
    ref = orc.hvp_x(C, inp["X"], inp["a"], inp["b"], eps, f.astype(np.float64),
                    g.astype(np.float64), inp["Y"], V)
    assert rel_l2(np64(hv), ref) <= APPLY_TOL


def test_hvp_symmetric_on_gpu():
    n, m, d, eps = 320, 256, 3, 0.15
    inp, C, f, g = _converged(n, m, d, 777, eps)
    rng = np.random.default_rng(9)
    U = rng.standard_normal((n, d)).astype(np.float32)
    V = rng.standard_normal((n, d)).astype(np.float32)
    t = to_dev(dict(inp, f=f, g=g, U=U, V=V))
    hu = np64(fs.fs_hvp_x(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["U"]))
    hv = np64(fs.fs_hvp_x(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"]))
    lhs, rhs = float(np.sum(U * hv)), float(np.sum(V * hu))
    assert abs(lhs - rhs) <= 1e-3 * max(abs(lhs), abs(rhs))


def test_hvp_tensor_path_matches_oracle():
    """d = 32 runs the plan applications on the tensor cores (split-precision
    scores, fp16 plan entries): the plan-application tolerance still holds."""
    n, m, d, eps = 400, 360, 32, 0.2
    inp, C, f, g = _converged(n, m, d, 612, eps)
    V = np.random.default_rng(32).standard_normal((n, d)).astype(np.float32)
    t = to_dev(dict(inp, f=f, g=g, V=V))
    hv = fs.fs_hvp_x(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"])
    ref = orc.hvp_x(C, inp["X"], inp["a"], inp["b"], eps, f.astype(np.float64),
                    g.astype(np.float64), inp["Y"], V)
    assert rel_l2(np64(hv), ref) <= APPLY_TOL


def _converged_recipe(name, n, m, d, eps, iters=2000):
    inp = make_inputs(name, n=n, m=m, d=d)
    C = orc.cost(inp["X"], inp["Y"])
    f, g = orc.sinkhorn(C, inp["a"], inp["b"], eps, iters)
    return inp, C, f.astype(np.float32), g.astype(np.float32)


@pytest.mark.parametrize("name,n,m,d,eps", [("c4_n50k_d512", 300, 280, 512, 0.1),
                                            ("c5_n20k_m30k_d1024", 200, 260, 1024, 0.2),
                                            ("c3_n50k_d64", 260, 300, 100, 0.05),
                                            ("c2_n10k_d3", 280, 250, 16, 0.05)])
def test_hvp_any_dimension_matches_oracle(name, n, m, d, eps):
    """The streamed HVP at the benchmark's dimensions (d = 512 and 1024 on the
    CTA-pair tensor path, d = 100 with a ragged second K chunk, d = 16 on the
    FMA path): O((n + m) d) scratch, the term sum_j P_ij Cdot_ij y_j from one
    tangent application, against the dense float64 least-squares oracle."""
    inp, C, f, g = _converged_recipe(name, n, m, d, eps)
    V = np.random.default_rng(d).standard_normal((n, d)).astype(np.float32)
    t = to_dev(dict(inp, f=f, g=g, V=V))
    hv = fs.fs_hvp_x(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"])
    ref = orc.hvp_x(C, inp["X"], inp["a"], inp["b"], eps, f.astype(np.float64),
                    g.astype(np.float64), inp["Y"], V)
    assert rel_l2(np64(hv), ref) <= APPLY_TOL


def test_hvp_tensor_path_forced_splits_and_host_buffers():
    """Column splits of the tangent application (partials merged in order)
    and host arrays staged through the library give the same HVP."""
    n, m, d, eps = 300, 900, 200, 0.2
    inp, C, f, g = _converged_recipe("c4_n50k_d512", n, m, d, eps)
    V = np.random.default_rng(4).standard_normal((n, d)).astype(np.float32)
    t = to_dev(dict(inp, f=f, g=g, V=V))
    ref = orc.hvp_x(C, inp["X"], inp["a"], inp["b"], eps, f.astype(np.float64),
                    g.astype(np.float64), inp["Y"], V)
    for splits in (1, 3):
        hv = fs.fs_hvp_x(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"],
                         splits=splits)
        assert rel_l2(np64(hv), ref) <= APPLY_TOL
    hh = fs.fs_hvp_x(inp["X"], inp["a"], inp["Y"], inp["b"], eps, f, g, V)
    assert rel_l2(np.asarray(hh, np.float64), ref) <= APPLY_TOL
