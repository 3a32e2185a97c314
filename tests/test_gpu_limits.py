"""Parity at the declared limits: the largest dimension (d = 4096, where Q no
longer stays in shared memory and is streamed beside K), a single row or
column against thousands, and the widest plan application (k = 4096)."""
import numpy as np
import pytest

import oracle as orc
from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import random_cloud
from tests.gpu_util import APPLY_TOL, F_TOL_TENSOR, max_abs, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


@pytest.mark.parametrize("n,m,d", [(130, 140, 4096), (70, 90, 2000), (1, 5000, 64),
                                   (5000, 1, 200), (3, 2049, 33)])
def test_tensor_path_extremes(n, m, d):
    inp = random_cloud(n, m, d, seed=1200 + d + n, spread=1.0 / np.sqrt(d), weights="lognormal")
    C = orc.cost(inp["X"], inp["Y"])
    eps = 0.05 * C.max()
    t = to_dev(inp)
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, 8, path="tensor")
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, 8)
    assert max_abs(np64(f), fr) <= F_TOL_TENSOR * C.max()
    assert max_abs(np64(g), gr) <= F_TOL_TENSOR * C.max()


@pytest.mark.parametrize("d,path", [(3, "fma"), (64, "tensor")])
def test_widest_plan_application(d, path):
    n, m, k = 300, 260, 4096
    inp = random_cloud(n, m, d, seed=1300 + d, spread=1.0 / np.sqrt(d), weights="lognormal")
    C = orc.cost(inp["X"], inp["Y"])
    eps = 0.1 * C.max()
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, 5)
    f32, g32 = fr.astype(np.float32), gr.astype(np.float32)
    V = np.random.default_rng(k + d).standard_normal((m, k)).astype(np.float32)
    t = to_dev(dict(inp, f=f32, g=g32, V=V))
    out = fs.fs_apply_plan(t["X"], t["a"], t["Y"], t["b"], eps, t["f"], t["g"], t["V"], path=path)
    ref = orc.apply_plan(C, inp["a"], inp["b"], eps, f32, g32, V)
    assert rel_l2(np64(out), ref) <= APPLY_TOL
