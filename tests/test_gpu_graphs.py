"""The solve and the plan operators captured into a CUDA graph and replayed
give the eager results bit for bit (the kernels are deterministic), on both
paths; capture refuses what it cannot hold."""
import numpy as np
import pytest

from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import random_cloud
from tests.gpu_util import np64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


@pytest.mark.parametrize("d,n,m", [(3, 3000, 2800), (64, 3000, 2800), (3, 16400, 16400)])
def test_solve_and_apply_replay_bitwise(d, n, m):
    """(3, 16400, 16400): 2.7e8 score pairs, so the captured solve includes
    the Morton sort, the per-CTA offset fits and the scatter back."""
    import torch
    inp = random_cloud(n, m, d, seed=900 + d, spread=1.0 / np.sqrt(d), weights="lognormal")
    t = to_dev(inp)
    eps, iters = 0.05, 12
    fe, ge = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, iters)   # also sizes
    oe = fs.fs_grad_x(t["X"], t["a"], t["Y"], t["b"], eps, fe, ge)              # the workspace
    torch.cuda.synchronize()

    f = torch.empty(n, device="cuda")
    g = torch.zeros(m, device="cuda")
    out = torch.empty(n, d, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, iters, f, g)
        fs.fs_grad_x(t["X"], t["a"], t["Y"], t["b"], eps, f, g, out)
    for _ in range(2):
        g.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(np64(f), np64(fe)) and np.array_equal(np64(g), np64(ge))
        assert np.array_equal(np64(out), np64(oe))


def test_capture_refuses_host_arrays_and_growth():
    import torch
    inp = random_cloud(500, 400, 3, seed=950)
    t = to_dev(inp)
    # earlier tests in the same process may have grown the workspace past
    # what the large problem below needs: start from an empty one
    torch.cuda.synchronize()
    fs.fs_release()
    fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], 0.1, 2)
    graph = torch.cuda.CUDAGraph()
    with pytest.raises(fs.FlashSinkhornError) as host_err:
        with torch.cuda.graph(graph):
            fs.fs_sinkhorn_solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.1, 2)
    assert host_err.value.status == fs.FS_ERR_UNSUPPORTED
    big = random_cloud(60000, 60000, 3, seed=951)
    tb = to_dev(big)
    graph2 = torch.cuda.CUDAGraph()
    with pytest.raises(fs.FlashSinkhornError) as grow_err:
        with torch.cuda.graph(graph2):
            fs.fs_sinkhorn_solve(tb["X"], tb["a"], tb["Y"], tb["b"], 0.1, 2)
    assert grow_err.value.status == fs.FS_ERR_UNSUPPORTED
