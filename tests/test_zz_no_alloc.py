"""The allocation-free solve (fs_sinkhorn_solve_noalloc) against the regular
entry point.

That entry point serves callers who may not allocate device memory, such as
a process whose device memory budget belongs to someone else or a loop where
the synchronisation of cudaMalloc/cudaFree is not allowed: its scratch is
one static array in the library's device image.  Two calls in a row must
each give the regular solve's potentials (the array is shared and reused),
within the FMA-path tolerance of 1e-4 max(C); at 2^26 score pairs, where the
regular solve takes reference offsets and the allocation-free one keeps the
online max, both are also checked against the float64 oracle.  The file sorts last so that
a run stopping at the first failure has run every other test first; it
also passes on its own in a fresh process.
"""
import numpy as np
import pytest

from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import make_inputs, random_cloud
from tests.gpu_util import F_TOL_FMA, max_abs, np64, to_dev

pytestmark = pytest.mark.gpu


def _cmax(inp):
    X = inp["X"].astype(np.float64)
    Y = inp["Y"].astype(np.float64)
    sx = (X * X).sum(1)[:, None]
    sy = (Y * Y).sum(1)[None, :]
    return float((sx + sy - 2 * X @ Y.T).max())


def _both(inp, eps, iters):
    import torch
    t = to_dev(inp)
    f_ref, g_ref = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, iters, path="fma")
    f = torch.empty_like(f_ref)
    g = torch.zeros_like(g_ref)
    fs.fs_sinkhorn_solve_noalloc(t["X"], t["a"], t["Y"], t["b"], eps, iters, f, g)
    torch.cuda.synchronize()
    return np64(f), np64(g), np64(f_ref), np64(g_ref)


def test_noalloc_matches_regular_solve_on_two_calls_in_a_row():
    fs.load_library()
    first = make_inputs("c1_n512_d2")
    second = random_cloud(3001, 2500, 3, seed=77, weights="lognormal")
    for inp, eps, iters in [(first, 0.05, 100), (second, 0.05, 40)]:
        f, g, fr, gr = _both(inp, eps, iters)
        tol = F_TOL_FMA * _cmax(inp)
        assert max_abs(f, fr) <= tol
        assert max_abs(g, gr) <= tol


def test_noalloc_at_2_26_pairs_matches_the_oracle_and_the_regular_solve():
    """n = m = 8192, d = 3 (2^26 score pairs): here the regular solve switches
    to reference offsets with fixups after two iterations, while the
    allocation-free one keeps the online max throughout, so the two run
    different kernels.  Both must match the float64 oracle element by element
    within 1e-4 max(C), on two allocation-free calls in a row."""
    import oracle as orc
    fs.load_library()
    inp = make_inputs("c2_n10k_d3", n=8192, m=8192, seed=405)
    eps, iters = 0.01, 12
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], eps, iters)
    tol = F_TOL_FMA * C.max()
    del C
    for _ in range(2):
        f, g, f_reg, g_reg = _both(inp, eps, iters)
        assert max_abs(f, fr) <= tol and max_abs(g, gr) <= tol
        assert max_abs(f_reg, fr) <= tol and max_abs(g_reg, gr) <= tol
        assert max_abs(f, f_reg) <= tol and max_abs(g, g_reg) <= tol


def test_noalloc_rejects_sizes_beyond_its_static_scratch():
    import torch
    fs.load_library()
    n = 32769
    X = torch.zeros(n, 2, device="cuda")
    a = torch.full((n,), 1.0 / n, device="cuda")
    Y = torch.zeros(10, 2, device="cuda")
    b = torch.full((10,), 0.1, device="cuda")
    f = torch.empty(n, device="cuda")
    g = torch.zeros(10, device="cuda")
    with pytest.raises(fs.FlashSinkhornError) as ei:
        fs.fs_sinkhorn_solve_noalloc(X, a, Y, b, 0.1, 1, f, g)
    assert ei.value.status == fs.FS_ERR_INVALID_ARG
    assert "32768" in str(ei.value)
