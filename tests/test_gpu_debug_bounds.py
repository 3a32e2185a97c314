"""Memory-safety check without a sanitizer: the debug build of the library
(FS_DEBUG_BOUNDS, libflashsinkhorn_dbg.so) tests the global-memory indices of
its FMA, preparation and block-sparse kernels against their buffers, records
the first index outside (and skips that access) instead of faulting.  Ragged
and edge-case problems run through it must record nothing, and still match
the float64 oracle.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle as orc
import oracle.block_sparse as bsp
from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import make_inputs, random_cloud
from tests.gpu_util import APPLY_TOL, F_TOL_FMA, max_abs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    import torch
    assert torch.cuda.is_available()
    if not os.path.exists(fs.DEBUG_LIB_PATH):
        from streaming_sinkhorn_solver_gb300.build import build
        build(debug_bounds=True)
    lib = fs.load_library(fs.DEBUG_LIB_PATH)
    en, word = ctypes.c_int32(), ctypes.c_uint64()
    assert lib.fs_debug_bounds(ctypes.byref(en), ctypes.byref(word)) == 0
    assert en.value == 1
    return lib


def _report(lib):
    import torch
    torch.cuda.synchronize()
    en, word = ctypes.c_int32(), ctypes.c_uint64()
    assert lib.fs_debug_bounds(ctypes.byref(en), ctypes.byref(word)) == 0
    return word.value


def _dev(inp):
    import torch
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in inp.items()}


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("n,m,d,splits", [(1, 1, 1, 0), (7, 300, 2, 0), (1025, 700, 3, 3),
                                          (1500, 1001, 8, 0), (513, 2049, 16, 5)])
def test_fma_solve_and_apply_record_no_bad_index(dbg, n, m, d, splits):
    import torch
    inp = random_cloud(n, m, d, seed=n + d, weights="lognormal")
    t = _dev(inp)
    f = torch.zeros(n, device="cuda")
    g = torch.zeros(m, device="cuda")
    opt = fs.fs_options()
    opt.path, opt.splits = 1, splits
    st = dbg.fs_sinkhorn_solve(_p(t["X"]), _p(t["a"]), n, _p(t["Y"]), _p(t["b"]), m, d,
                               ctypes.c_float(0.1), 6, _p(f), _p(g), ctypes.byref(opt), None)
    assert st == 0
    out = torch.empty(n, d, device="cuda")
    st = dbg.fs_apply_plan(_p(t["X"]), _p(t["a"]), n, _p(t["Y"]), _p(t["b"]), m, d,
                           ctypes.c_float(0.1), _p(f), _p(g), _p(t["Y"]), d, _p(out),
                           ctypes.byref(opt), None)
    assert st == 0
    assert _report(dbg) == 0
    C = orc.cost(inp["X"], inp["Y"])
    fr, gr = orc.sinkhorn(C, inp["a"], inp["b"], 0.1, 6)
    assert max_abs(f.cpu().numpy(), fr) <= F_TOL_FMA * C.max()
    ref = orc.apply_plan(C, inp["a"], inp["b"], 0.1, f.cpu().numpy(), g.cpu().numpy(), inp["Y"])
    assert rel_l2(out.cpu().numpy(), ref) <= APPLY_TOL


@pytest.mark.parametrize("n,m,d,tau,online", [(1, 1, 1, 1e-6, 0), (300, 129, 2, 1e-5, -1),
                                              (2049, 1900, 3, 1e-6, -1), (3000, 2600, 2, 1e-4, 0),
                                              (700, 513, 4, 1e-5, -1), (1100, 900, 5, 1e-6, 0),
                                              (1300, 1029, 8, 1e-5, -1), (1, 2, 8, 1e-6, 0),
                                              # >= 32 input blocks: the super-block cull and
                                              # kept-list rows sized by its survivors
                                              (6000, 5200, 3, 1e-6, -1), (5000, 4600, 5, 1e-5, 0)])
def test_block_sparse_solve_records_no_bad_index(dbg, n, m, d, tau, online):
    import torch
    inp = make_inputs("c2_n10k_d3", n=n, m=m, d=d)
    t = _dev(inp)
    f = torch.zeros(n, device="cuda")
    g = torch.zeros(m, device="cuda")
    o = fs.fs_sparse_options()
    o.coarse_iters, o.max_iters, o.tau, o.online_iters = 3, 6, tau, online
    o.target, o.check_every = 1e-9, 2
    o.lift_samples, o.lift_rounds, o.lift_tol = 77, 1, 0.0     # one extra centroid round
    rep = fs.fs_sparse_report()
    st = dbg.fs_sparse_solve(_p(t["X"]), _p(t["a"]), n, _p(t["Y"]), _p(t["b"]), m, d,
                             ctypes.c_float(0.005), ctypes.byref(o), _p(f), _p(g),
                             ctypes.byref(rep), None)
    assert st == 0, dbg.fs_last_error()
    assert _report(dbg) == 0
    fr, gr, _ = bsp.solve(inp["X"], inp["a"], inp["Y"], inp["b"], 0.005, 3, 6, tau,
                          target=1e-9, check_every=2, lift_samples=77, lift_tol=0.0,
                          lift_rounds=1)
    C = orc.cost(inp["X"], inp["Y"])
    assert max_abs(f.cpu().numpy(), fr) <= F_TOL_FMA * C.max()
