"""The C-ABI library loads, exports every symbol include/*.h declares, and
rejects bad arguments on the host before touching the GPU (no compute calls
here: these run without a GPU)."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

from streaming_sinkhorn_solver_gb300 import binding as fs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for mname in re.finditer(r"\b(fs_[a-z0-9_]+)\s*\(", text):
            names.add(mname.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from streaming_sinkhorn_solver_gb300.build import build
    build()
    return fs.load_library()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("fs_sinkhorn_solve", "fs_apply_plan", "fs_grad_x", "fs_barycentric",
                     "fs_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(_declared_functions()) <= set(fs.EXPORTED)


def test_version_and_launch_counter(lib):
    assert re.match(r"^\d+\.\d+\.\d+$", fs.fs_version())
    assert fs.fs_launch_count() >= 0


def _small():
    X = np.zeros((4, 2), np.float32)
    Y = np.zeros((5, 2), np.float32)
    a = np.full(4, 0.25, np.float32)
    b = np.full(5, 0.2, np.float32)
    return X, a, Y, b


@pytest.mark.parametrize("bad", ["eps0", "epsnan", "iters0", "path", "reserved", "splits",
                                 "row_shards"])
def test_invalid_arguments_rejected_on_host(lib, bad):
    X, a, Y, b = _small()
    f = np.zeros(4, np.float32)
    g = np.zeros(5, np.float32)
    opt = fs.fs_options()
    eps, iters = 0.1, 3
    if bad == "eps0":
        eps = 0.0
    elif bad == "epsnan":
        eps = float("nan")
    elif bad == "iters0":
        iters = 0
    elif bad == "path":
        opt.path = 7
    elif bad == "reserved":
        opt.reserved[2] = 1
    elif bad == "splits":
        opt.splits = -1
    elif bad == "row_shards":
        opt.row_shards = -2
    st = lib.fs_sinkhorn_solve(X.ctypes.data, a.ctypes.data, 4, Y.ctypes.data, b.ctypes.data, 5, 2,
                               eps, iters, f.ctypes.data, g.ctypes.data, ctypes.byref(opt), None)
    assert st == fs.FS_ERR_INVALID_ARG
    assert fs.fs_last_error()


def test_bad_sizes_and_null_pointers(lib):
    X, a, Y, b = _small()
    f = np.zeros(4, np.float32)
    g = np.zeros(5, np.float32)
    for n, m, d in [(0, 5, 2), (4, 0, 2), (4, 5, 0), (4, 5, 5000)]:
        st = lib.fs_sinkhorn_solve(X.ctypes.data, a.ctypes.data, n, Y.ctypes.data, b.ctypes.data,
                                   m, d, 0.1, 1, f.ctypes.data, g.ctypes.data, None, None)
        assert st == fs.FS_ERR_INVALID_ARG
    st = lib.fs_sinkhorn_solve(None, a.ctypes.data, 4, Y.ctypes.data, b.ctypes.data, 5, 2, 0.1, 1,
                               f.ctypes.data, g.ctypes.data, None, None)
    assert st == fs.FS_ERR_INVALID_ARG
    out = np.zeros((4, 3), np.float32)
    V = np.zeros((5, 3), np.float32)
    st = lib.fs_apply_plan(X.ctypes.data, a.ctypes.data, 4, Y.ctypes.data, b.ctypes.data, 5, 2,
                           0.1, f.ctypes.data, g.ctypes.data, V.ctypes.data, 0, out.ctypes.data,
                           None, None)
    assert st == fs.FS_ERR_INVALID_ARG


def test_fma_path_rejects_large_d(lib):
    X = np.zeros((4, 17), np.float32)
    Y = np.zeros((5, 17), np.float32)
    a = np.full(4, 0.25, np.float32)
    b = np.full(5, 0.2, np.float32)
    with pytest.raises(fs.FlashSinkhornError) as ei:
        fs.fs_sinkhorn_solve(X, a, Y, b, 0.1, 1, path="fma")
    assert ei.value.status == fs.FS_ERR_UNSUPPORTED


def test_binding_rejects_wrong_dtype_and_layout(lib):
    X, a, Y, b = _small()
    with pytest.raises(TypeError):
        fs.fs_sinkhorn_solve(X.astype(np.float64), a, Y, b, 0.1, 1)
    with pytest.raises(TypeError):
        fs.fs_sinkhorn_solve(np.asfortranarray(np.zeros((4, 3), np.float32)), a,
                             np.zeros((5, 3), np.float32), b, 0.1, 1)
    with pytest.raises(ValueError):
        fs.fs_sinkhorn_solve(X, a[:3], Y, b, 0.1, 1)


def test_workspace_is_linear_in_sizes(lib):
    w1 = fs.fs_workspace_bytes(10_000, 10_000, 3)
    w2 = fs.fs_workspace_bytes(20_000, 20_000, 3)
    assert 0 < w1 < w2 < 3 * w1
    # no n x m buffer: far below n*m*4 bytes at 50k
    assert fs.fs_workspace_bytes(50_000, 50_000, 3) < 50_000 * 50_000 * 4 // 100


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        fs.load_library(str(tmp_path / "nope.so"))


def test_y_side_and_reports_reject_bad_arguments(lib):
    X, a, Y, b = _small()
    f = np.zeros(4, np.float32)
    g = np.zeros(5, np.float32)
    U = np.zeros((4, 3), np.float32)
    out = np.zeros((5, 3), np.float32)
    st = lib.fs_apply_plan_t(X.ctypes.data, a.ctypes.data, 4, Y.ctypes.data, b.ctypes.data, 5, 2,
                             0.1, f.ctypes.data, g.ctypes.data, U.ctypes.data, 0, out.ctypes.data,
                             None, None)
    assert st == fs.FS_ERR_INVALID_ARG
    st = lib.fs_grad_y(X.ctypes.data, a.ctypes.data, 4, Y.ctypes.data, b.ctypes.data, 5, 2, 0.0,
                       f.ctypes.data, g.ctypes.data, out.ctypes.data, None, None)
    assert st == fs.FS_ERR_INVALID_ARG
    res = (ctypes.c_double * 2)()
    st = lib.fs_dual_value(None, 4, b.ctypes.data, 5, f.ctypes.data, g.ctypes.data, res, None)
    assert st == fs.FS_ERR_INVALID_ARG
    st = lib.fs_dual_value(a.ctypes.data, 0, b.ctypes.data, 5, f.ctypes.data, g.ctypes.data, res,
                           None)
    assert st == fs.FS_ERR_INVALID_ARG
    st = lib.fs_marginal_residuals(X.ctypes.data, a.ctypes.data, 4, Y.ctypes.data, b.ctypes.data,
                                   5, 2, 0.1, f.ctypes.data, g.ctypes.data, None, None, None)
    assert st == fs.FS_ERR_INVALID_ARG


def test_hvp_rejects_bad_arguments(lib):
    X, a, Y, b = _small()
    f = np.zeros(4, np.float32)
    g = np.zeros(5, np.float32)
    V = np.zeros((4, 2), np.float32)
    out = np.zeros((4, 2), np.float32)
    st = lib.fs_hvp_x(X.ctypes.data, a.ctypes.data, 4, Y.ctypes.data, b.ctypes.data, 5, 2, 0.1,
                      f.ctypes.data, g.ctypes.data, None, out.ctypes.data, 0, 0.0, None, None)
    assert st == fs.FS_ERR_INVALID_ARG
    st = lib.fs_hvp_x(X.ctypes.data, a.ctypes.data, 4, Y.ctypes.data, b.ctypes.data, 5, 5000, 0.1,
                      f.ctypes.data, g.ctypes.data, V.ctypes.data, out.ctypes.data, 0, 0.0, None,
                      None)
    assert st == fs.FS_ERR_INVALID_ARG
    opt = fs.fs_options()
    opt.cost = fs.COSTS["cosine"]
    st = lib.fs_hvp_x(X.ctypes.data, a.ctypes.data, 4, Y.ctypes.data, b.ctypes.data, 5, 2, 0.1,
                      f.ctypes.data, g.ctypes.data, V.ctypes.data, out.ctypes.data, 0, 0.0,
                      ctypes.byref(opt), None)
    assert st == fs.FS_ERR_UNSUPPORTED


_CTYPE = {"int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64, "float": ctypes.c_float,
          "double": ctypes.c_double}


def _header_structs():
    """{struct name: [(field, C type, array length or 0), ...]} from include/*.h."""
    out = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for mt in re.finditer(r"typedef\s+struct\s+(\w+)\s*\{(.*?)\}\s*(\w+)\s*;", text, flags=re.S):
            fields = []
            for decl in mt.group(2).split(";"):
                decl = decl.strip()
                if not decl:
                    continue
                ctype, names = decl.split(None, 1)
                for name in names.split(","):
                    name = name.strip()
                    arr = re.match(r"(\w+)\[(\d+)\]", name)
                    fields.append((arr.group(1), ctype, int(arr.group(2))) if arr else (name, ctype, 0))
            out[mt.group(3)] = fields
    return out


@pytest.mark.parametrize("name", ["fs_options", "fs_sparse_options", "fs_sparse_report"])
def test_binding_structs_mirror_the_header(name):
    """The ctypes structures of the binding have the header's fields, in
    order, with the same types and array lengths, so they have its layout."""
    want = _header_structs()[name]
    got = getattr(fs, name)._fields_
    assert [f for f, _ in got] == [f for f, _, _ in want]
    for (fname, ctype_b), (_, ctype_h, n) in zip(got, want):
        ref = _CTYPE[ctype_h] * n if n else _CTYPE[ctype_h]
        assert ctypes.sizeof(ctype_b) == ctypes.sizeof(ref), fname
        base = ctype_b._type_ if hasattr(ctype_b, "_length_") else ctype_b
        assert base == _CTYPE[ctype_h], fname
        assert getattr(ctype_b, "_length_", 0) == n, fname


def _header_functions():
    """{name: (return type, parameter count)} of the functions include/*.h declares."""
    out = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for mt in re.finditer(r"([A-Za-z_][\w\s\*]*?)\b(fs_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
            ret = " ".join(mt.group(1).split())
            params = " ".join(mt.group(3).split())
            n = 0 if params in ("", "void") else params.count(",") + 1
            out[mt.group(2)] = (ret, n)
    return out


def test_binding_declares_every_signature(lib):
    """Every declared function has ctypes argtypes of the header's arity and
    a restype of the header's width (an unset argtypes would pass 64-bit
    pointers and sizes as C ints)."""
    funcs = _header_functions()
    assert "fs_sinkhorn_solve" in funcs and "fs_shard_range" in funcs
    for name, (ret, n) in funcs.items():
        fn = getattr(lib, name)
        if n:
            assert fn.argtypes is not None and len(fn.argtypes) == n, name
        if ret.endswith("fs_status"):
            assert fn.restype in (ctypes.c_int, ctypes.c_int32), name
        elif ret.endswith("int64_t"):
            assert fn.restype == ctypes.c_int64, name
        elif ret.endswith("char*") or ret.endswith("char *"):
            assert fn.restype == ctypes.c_char_p, name


def test_hvp_workspace_is_linear_in_the_dimension(lib):
    """fs_hvp_x keeps O((n + m) d) device memory: no n x m array and no
    n d^2 products (doubling d at most doubles it, doubling n and m at most
    doubles it)."""
    for d in (64, 512, 1024):
        b1 = fs.fs_hvp_workspace_bytes(20000, 30000, d)
        assert b1 > 0
        assert fs.fs_hvp_workspace_bytes(20000, 30000, 2 * d) <= 2.05 * b1
        assert fs.fs_hvp_workspace_bytes(40000, 60000, d) <= 2.5 * b1
    # far below n d^2 floats at d = 1024
    assert fs.fs_hvp_workspace_bytes(50000, 50000, 1024) < 4 * 50000 * 1024 * 64
    assert fs.fs_hvp_workspace_bytes(100, 100, 8, path="fma") > 0
