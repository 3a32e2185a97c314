"""ctypes binding of libflashsinkhorn (include/flashsinkhorn.h).

Argument marshalling only: every function passes pointers, sizes and the
current CUDA stream to the C ABI function of the same name, and every step
of the computation runs in the library's CUDA kernels.  Arrays are float32,
C-contiguous torch tensors (CUDA or CPU) or numpy arrays; CPU arrays are
staged by the library itself.  Nothing is converted silently: a wrong dtype,
layout or shape raises before the call.

The library must have been built (``python -m streaming_sinkhorn_solver_gb300.build``
or ``__graft_entry__.build()``); if it is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libflashsinkhorn.so")
# debug build with global-memory index checks (build(debug_bounds=True))
DEBUG_LIB_PATH = os.path.join(_HERE, "libflashsinkhorn_dbg.so")

FS_OK, FS_ERR_INVALID_ARG, FS_ERR_CUDA, FS_ERR_OOM = 0, 1, 2, 3
FS_ERR_NONFINITE, FS_ERR_TIMEOUT, FS_ERR_UNSUPPORTED = 4, 5, 6
_STATUS = {0: "FS_OK", 1: "FS_ERR_INVALID_ARG", 2: "FS_ERR_CUDA", 3: "FS_ERR_OOM",
           4: "FS_ERR_NONFINITE", 5: "FS_ERR_TIMEOUT", 6: "FS_ERR_UNSUPPORTED"}
PATHS = {"auto": 0, "fma": 1, "tensor": 2}

EXPORTED = ("fs_sinkhorn_solve", "fs_apply_plan", "fs_barycentric", "fs_grad_x",
            "fs_apply_plan_t", "fs_barycentric_y", "fs_grad_y", "fs_dual_value",
            "fs_marginal_residuals", "fs_workspace_bytes", "fs_check", "fs_release",
            "fs_last_error", "fs_version", "fs_launch_count", "fs_timing_enable",
            "fs_timing_read", "fs_sinkhorn_solve_noalloc", "fs_unit_rates", "fs_hvp_x",
            "fs_sparse_solve", "fs_morton_order", "fs_sparse_screen", "fs_wait_selftest",
            "fs_debug_bounds", "fs_shard_unit", "fs_shard_range", "fs_fixup_stats",
            "fs_hvp_workspace_bytes", "fs_barrier_selftest")


class FlashSinkhornError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


COSTS = {"sqeuclidean": 0, "cosine": 1}


class fs_options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("check_finite", ctypes.c_int32), ("cost", ctypes.c_int32),
                ("row_shards", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]


class fs_sparse_options(ctypes.Structure):
    _fields_ = [("coarse_iters", ctypes.c_int32), ("max_iters", ctypes.c_int32),
                ("check_every", ctypes.c_int32), ("tau", ctypes.c_float),
                ("target", ctypes.c_float), ("online_iters", ctypes.c_int32),
                ("lift_samples", ctypes.c_int32), ("lift_rounds", ctypes.c_int32),
                ("lift_tol", ctypes.c_float)]


class fs_sparse_report(ctypes.Structure):
    _fields_ = [("iters", ctypes.c_int32), ("passes", ctypes.c_int32),
                ("blocks_x", ctypes.c_int32), ("blocks_y", ctypes.c_int32),
                ("residual", ctypes.c_double), ("kept_blocks", ctypes.c_double),
                ("kept_pairs", ctypes.c_double), ("exact_bounds", ctypes.c_double),
                ("fixed_rows", ctypes.c_double), ("lift_checks", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("lift_error", ctypes.c_double)]


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[str] = None):
    """Load (once) and return the ctypes handle; raises if the .so is absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} is missing: build it with "
                              "'python -m streaming_sinkhorn_solver_gb300.build'")
        lib = ctypes.CDLL(p)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        opt = ctypes.POINTER(fs_options)
        lib.fs_sinkhorn_solve.argtypes = [vp, vp, i64, vp, vp, i64, i32, f32, i32, vp, vp, opt, vp]
        lib.fs_apply_plan.argtypes = [vp, vp, i64, vp, vp, i64, i32, f32, vp, vp, vp, i32, vp, opt, vp]
        lib.fs_barycentric.argtypes = [vp, vp, i64, vp, vp, i64, i32, f32, vp, vp, vp, opt, vp]
        lib.fs_grad_x.argtypes = [vp, vp, i64, vp, vp, i64, i32, f32, vp, vp, vp, opt, vp]
        lib.fs_apply_plan_t.argtypes = lib.fs_apply_plan.argtypes
        lib.fs_barycentric_y.argtypes = lib.fs_barycentric.argtypes
        lib.fs_grad_y.argtypes = lib.fs_grad_x.argtypes
        lib.fs_dual_value.argtypes = [vp, i64, vp, i64, vp, vp, ctypes.POINTER(ctypes.c_double), vp]
        lib.fs_marginal_residuals.argtypes = [vp, vp, i64, vp, vp, i64, i32, f32, vp, vp,
                                              ctypes.POINTER(ctypes.c_double), opt, vp]
        for fn in ("fs_sinkhorn_solve", "fs_apply_plan", "fs_barycentric", "fs_grad_x",
                   "fs_apply_plan_t", "fs_barycentric_y", "fs_grad_y", "fs_dual_value",
                   "fs_marginal_residuals", "fs_check", "fs_release"):
            getattr(lib, fn).restype = ctypes.c_int
        lib.fs_workspace_bytes.argtypes = [i64, i64, i32, i32, opt]
        lib.fs_workspace_bytes.restype = i64
        lib.fs_check.argtypes = [vp]
        lib.fs_release.argtypes = []
        lib.fs_last_error.restype = ctypes.c_char_p
        lib.fs_version.restype = ctypes.c_char_p
        lib.fs_launch_count.restype = i64
        lib.fs_timing_enable.argtypes = [i32]
        lib.fs_timing_enable.restype = ctypes.c_int
        lib.fs_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]
        lib.fs_timing_read.restype = ctypes.c_int
        lib.fs_sinkhorn_solve_noalloc.argtypes = [vp, vp, i64, vp, vp, i64, i32, f32, i32, vp, vp, vp]
        lib.fs_sinkhorn_solve_noalloc.restype = ctypes.c_int
        lib.fs_hvp_x.argtypes = [vp, vp, i64, vp, vp, i64, i32, f32, vp, vp, vp, vp, i32, f32,
                                 opt, vp]
        lib.fs_hvp_x.restype = ctypes.c_int
        lib.fs_unit_rates.argtypes = [ctypes.POINTER(ctypes.c_double), vp]
        lib.fs_unit_rates.restype = ctypes.c_int
        lib.fs_sparse_solve.argtypes = [vp, vp, i64, vp, vp, i64, i32, f32,
                                        ctypes.POINTER(fs_sparse_options), vp, vp,
                                        ctypes.POINTER(fs_sparse_report), vp]
        lib.fs_sparse_solve.restype = ctypes.c_int
        lib.fs_morton_order.argtypes = [vp, i64, vp, i64, i32, vp, vp, vp]
        lib.fs_morton_order.restype = ctypes.c_int
        lib.fs_sparse_screen.argtypes = [vp, vp, i64, vp, vp, i64, i32, f32, vp, vp, f32, i32,
                                         vp, vp, vp]
        lib.fs_sparse_screen.restype = ctypes.c_int
        lib.fs_wait_selftest.argtypes = [i64, vp]
        lib.fs_wait_selftest.restype = ctypes.c_int
        lib.fs_debug_bounds.argtypes = [ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_uint64)]
        lib.fs_debug_bounds.restype = ctypes.c_int
        lib.fs_shard_unit.argtypes = [i32, opt]
        lib.fs_shard_unit.restype = i64
        lib.fs_shard_range.argtypes = [i64, i64, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.fs_shard_range.restype = ctypes.c_int
        lib.fs_fixup_stats.argtypes = [ctypes.POINTER(ctypes.c_uint64),
                                       ctypes.POINTER(ctypes.c_uint64), i32]
        lib.fs_fixup_stats.restype = ctypes.c_int
        lib.fs_hvp_workspace_bytes.argtypes = [i64, i64, i32, opt]
        lib.fs_hvp_workspace_bytes.restype = i64
        lib.fs_barrier_selftest.argtypes = [i64, vp]
        lib.fs_barrier_selftest.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


# ---------------------------------------------------------------------------
# marshalling helpers

def _is_torch(x) -> bool:
    return type(x).__module__.startswith("torch")


def _ptr(x, name: str, shape) -> int:
    """Pointer of a float32 C-contiguous tensor/array with the given shape."""
    if _is_torch(x):
        import torch
        if x.dtype != torch.float32:
            raise TypeError(f"{name} must be float32, got {x.dtype}")
        if not x.is_contiguous():
            raise TypeError(f"{name} must be contiguous")
        if tuple(x.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(x.shape)}, expected {tuple(shape)}")
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        if x.dtype != np.float32:
            raise TypeError(f"{name} must be float32, got {x.dtype}")
        if not x.flags.c_contiguous:
            raise TypeError(f"{name} must be C-contiguous")
        if tuple(x.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(x.shape)}, expected {tuple(shape)}")
        return x.ctypes.data
    raise TypeError(f"{name} must be a torch tensor or numpy array, got {type(x).__name__}")


def _on_cuda(*xs) -> bool:
    return any(_is_torch(x) and x.is_cuda for x in xs)


def _stream(stream, *xs):
    """The cudaStream_t to use: explicit, else torch's current stream."""
    if stream is not None:
        return ctypes.c_void_p(int(getattr(stream, "cuda_stream", stream)))
    try:
        import torch
        if torch.cuda.is_available():
            return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    except Exception:
        pass
    return ctypes.c_void_p(0)


def _opts(path: str, splits: int, check_finite: bool, cost: str = "sqeuclidean",
          row_shards: int = 0):
    o = fs_options()
    o.path = PATHS[path]
    o.splits = int(splits)
    o.check_finite = 1 if check_finite else 0
    o.cost = COSTS[cost]
    o.row_shards = int(row_shards)
    return ctypes.byref(o)


def _raise(status: int):
    if status != FS_OK:
        msg = load_library().fs_last_error().decode(errors="replace")
        raise FlashSinkhornError(status, msg)


def _host_sync(stream, *xs):
    """Host outputs are valid once the stream is synchronised."""
    if not _on_cuda(*xs):
        try:
            import torch
            if torch.cuda.is_available():
                torch.cuda.synchronize()
        except Exception:
            pass


def _new_like(ref, shape):
    if _is_torch(ref):
        import torch
        return torch.empty(shape, dtype=torch.float32, device=ref.device)
    return np.empty(shape, dtype=np.float32)


def _zeros_like(ref, shape):
    if _is_torch(ref):
        import torch
        return torch.zeros(shape, dtype=torch.float32, device=ref.device)
    return np.zeros(shape, dtype=np.float32)


# ---------------------------------------------------------------------------
# the C ABI, one function each

def fs_sinkhorn_solve(X, a, Y, b, eps: float, n_iter: int, f=None, g=None, *, path: str = "auto", cost: str = "sqeuclidean",
                      splits: int = 0, check_finite: bool = False, row_shards: int = 0,
                      stream=None) -> Tuple:
    """n_iter log-domain Sinkhorn iterations; f, g are in/out (g seeds the first
    f-update, zeros if None).  Returns (f, g).  row_shards = G >= 2 runs every
    half-update as G row shards, one after the other (the per-GPU launches of
    a G-way row partition); the result is bitwise that of one launch."""
    n, d = X.shape
    m = Y.shape[0]
    f = _new_like(X, (n,)) if f is None else f
    g = _zeros_like(X, (m,)) if g is None else g
    st = load_library().fs_sinkhorn_solve(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), int(n_iter), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)),
        _opts(path, splits, check_finite, cost, row_shards), _stream(stream, X))
    _raise(st)
    _host_sync(stream, X, f, g)
    return f, g


def fs_shard_unit(d: int, path: str = "auto") -> int:
    """Rows per shard unit (the half-update's row block) for dimension d."""
    o = fs_options()
    o.path = PATHS[path]
    u = load_library().fs_shard_unit(int(d), ctypes.byref(o))
    if u < 1:
        raise FlashSinkhornError(1, f"no shard unit for d={d}, path={path}")
    return int(u)


def fs_shard_range(rows: int, unit: int, shards: int, s: int) -> Tuple[int, int]:
    """Row range [r0, r1) of shard s of `shards` (host only)."""
    r0, r1 = ctypes.c_int64(), ctypes.c_int64()
    _raise(load_library().fs_shard_range(int(rows), int(unit), int(shards), int(s),
                                         ctypes.byref(r0), ctypes.byref(r1)))
    return r0.value, r1.value


def fs_apply_plan(X, a, Y, b, eps: float, f, g, V, out=None, *, path: str = "auto", cost: str = "sqeuclidean",
                  splits: int = 0, check_finite: bool = False, stream=None):
    """out = P V with P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps); V is m x k."""
    n, d = X.shape
    m = Y.shape[0]
    squeeze = len(V.shape) == 1
    k = 1 if squeeze else V.shape[1]
    out = _new_like(X, (n, k) if not squeeze else (n,)) if out is None else out
    st = load_library().fs_apply_plan(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)),
        _ptr(V, "V", (m,) if squeeze else (m, k)), k,
        _ptr(out, "out", (n,) if squeeze else (n, k)),
        _opts(path, splits, check_finite, cost), _stream(stream, X))
    _raise(st)
    _host_sync(stream, X, out)
    return out


def fs_barycentric(X, a, Y, b, eps: float, f, g, out=None, *, path: str = "auto", cost: str = "sqeuclidean",
                   splits: int = 0, check_finite: bool = False, stream=None):
    """T_i = (P Y)_i / a_i."""
    n, d = X.shape
    m = Y.shape[0]
    out = _new_like(X, (n, d)) if out is None else out
    st = load_library().fs_barycentric(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)), _ptr(out, "out", (n, d)),
        _opts(path, splits, check_finite, cost), _stream(stream, X))
    _raise(st)
    _host_sync(stream, X, out)
    return out


def fs_grad_x(X, a, Y, b, eps: float, f, g, out=None, *, path: str = "auto", cost: str = "sqeuclidean", splits: int = 0,
              check_finite: bool = False, stream=None):
    """grad_i = 2 (a_i x_i - (P Y)_i)."""
    n, d = X.shape
    m = Y.shape[0]
    out = _new_like(X, (n, d)) if out is None else out
    st = load_library().fs_grad_x(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)), _ptr(out, "out", (n, d)),
        _opts(path, splits, check_finite, cost), _stream(stream, X))
    _raise(st)
    _host_sync(stream, X, out)
    return out


def fs_apply_plan_t(X, a, Y, b, eps: float, f, g, U, out=None, *, path: str = "auto", cost: str = "sqeuclidean",
                    splits: int = 0, check_finite: bool = False, stream=None):
    """out = P^T U (m x k); U is n x k."""
    n, d = X.shape
    m = Y.shape[0]
    squeeze = len(U.shape) == 1
    k = 1 if squeeze else U.shape[1]
    out = _new_like(Y, (m, k) if not squeeze else (m,)) if out is None else out
    st = load_library().fs_apply_plan_t(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)),
        _ptr(U, "U", (n,) if squeeze else (n, k)), k,
        _ptr(out, "out", (m,) if squeeze else (m, k)),
        _opts(path, splits, check_finite, cost), _stream(stream, X))
    _raise(st)
    _host_sync(stream, X, out)
    return out


def _y_side(fn, X, a, Y, b, eps, f, g, out, path, splits, check_finite, stream, cost="sqeuclidean"):
    n, d = X.shape
    m = Y.shape[0]
    out = _new_like(Y, (m, d)) if out is None else out
    st = getattr(load_library(), fn)(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)), _ptr(out, "out", (m, d)),
        _opts(path, splits, check_finite, cost), _stream(stream, X))
    _raise(st)
    _host_sync(stream, X, out)
    return out


def fs_barycentric_y(X, a, Y, b, eps: float, f, g, out=None, *, path: str = "auto", cost: str = "sqeuclidean",
                     splits: int = 0, check_finite: bool = False, stream=None):
    """T_j = (P^T X)_j / b_j."""
    return _y_side("fs_barycentric_y", X, a, Y, b, eps, f, g, out, path, splits, check_finite,
                   stream, cost)


def fs_grad_y(X, a, Y, b, eps: float, f, g, out=None, *, path: str = "auto", cost: str = "sqeuclidean", splits: int = 0,
              check_finite: bool = False, stream=None):
    """grad_j = 2 (b_j y_j - (P^T X)_j)."""
    return _y_side("fs_grad_y", X, a, Y, b, eps, f, g, out, path, splits, check_finite, stream,
                   cost)


def fs_dual_value(a, b, f, g, *, stream=None) -> float:
    """<a, f> + <b, g>, summed on the GPU in double."""
    n, m = a.shape[0], b.shape[0]
    out = ctypes.c_double(0.0)
    st = load_library().fs_dual_value(_ptr(a, "a", (n,)), n, _ptr(b, "b", (m,)), m,
                                      _ptr(f, "f", (n,)), _ptr(g, "g", (m,)), ctypes.byref(out),
                                      _stream(stream, a))
    _raise(st)
    return float(out.value)


def fs_marginal_residuals(X, a, Y, b, eps: float, f, g, *, path: str = "auto", cost: str = "sqeuclidean", splits: int = 0,
                          stream=None):
    """(||P 1 - a||_1, ||P^T 1 - b||_1)."""
    n, d = X.shape
    m = Y.shape[0]
    out = (ctypes.c_double * 2)()
    st = load_library().fs_marginal_residuals(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)), out, _opts(path, splits, False, cost),
        _stream(stream, X))
    _raise(st)
    return float(out[0]), float(out[1])


def fs_hvp_x(X, a, Y, b, eps: float, f, g, V, out=None, *, cg_max_iter: int = 0,
             cg_tol: float = 0.0, path: str = "auto", splits: int = 0, stream=None):
    """(H V), H the Hessian of the converged OT value with respect to X."""
    n, d = X.shape
    m = Y.shape[0]
    out = _new_like(X, (n, d)) if out is None else out
    st = load_library().fs_hvp_x(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)), _ptr(V, "V", (n, d)),
        _ptr(out, "out", (n, d)), int(cg_max_iter), float(cg_tol), _opts(path, splits, False),
        _stream(stream, X))
    _raise(st)
    return out


def fs_hvp_workspace_bytes(n: int, m: int, d: int, *, path: str = "auto") -> int:
    """Device bytes fs_hvp_x uses for these sizes (host only)."""
    return int(load_library().fs_hvp_workspace_bytes(n, m, d, _opts(path, 0, False)))


def fs_unit_rates(stream=None) -> dict:
    """Measured per-SM rates (results per clock per SM) and the SM count."""
    out = (ctypes.c_double * 5)()
    _raise(load_library().fs_unit_rates(out, _stream(stream)))
    return {"ex2_per_clk_sm": out[0], "fma2_lanes_per_clk_sm": out[1],
            "fma_per_clk_sm": out[2], "max3_per_clk_sm": out[3], "sms": int(out[4])}


def fs_workspace_bytes(n: int, m: int, d: int, k: int = 0, *, path: str = "auto", cost: str = "sqeuclidean",
                       splits: int = 0) -> int:
    return int(load_library().fs_workspace_bytes(n, m, d, k, _opts(path, splits, False, cost)))


def fs_check(stream=None) -> None:
    _raise(load_library().fs_check(_stream(stream)))


def fs_release() -> None:
    _raise(load_library().fs_release())


def fs_last_error() -> str:
    return load_library().fs_last_error().decode(errors="replace")


def fs_version() -> str:
    return load_library().fs_version().decode()


def fs_launch_count() -> int:
    return int(load_library().fs_launch_count())


def fs_fixup_stats(reset: bool = False):
    """(fixup launches, rows recomputed) of the reference-offset half-updates
    on the current device since the last reset (synchronises the device)."""
    launches, rows = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _raise(load_library().fs_fixup_stats(ctypes.byref(launches), ctypes.byref(rows),
                                         1 if reset else 0))
    return int(launches.value), int(rows.value)


def fs_timing_enable(on: bool = True) -> None:
    _raise(load_library().fs_timing_enable(1 if on else 0))


def fs_timing_read():
    """Returns ((half_ms, apply_ms, prep_ms), (half_n, apply_n, prep_n)) since the last read."""
    ms = (ctypes.c_double * 3)()
    cnt = (ctypes.c_int64 * 3)()
    _raise(load_library().fs_timing_read(ms, cnt))
    return (ms[0], ms[1], ms[2]), (int(cnt[0]), int(cnt[1]), int(cnt[2]))


def fs_sinkhorn_solve_noalloc(X, a, Y, b, eps: float, n_iter: int, f, g, *, stream=None):
    """The FMA-path solve with no device allocation (see the C header for
    who needs it and its limits).  Every array must be a CUDA tensor; f and g
    are in/out as in fs_sinkhorn_solve.  Returns (f, g)."""
    n, d = X.shape
    m = Y.shape[0]
    st = load_library().fs_sinkhorn_solve_noalloc(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), int(n_iter), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)), _stream(stream, X))
    _raise(st)
    return f, g


# ---------------------------------------------------------------------------
# block-sparse solver for low dimension (d <= 8)

def fs_sparse_solve(X, a, Y, b, eps: float, *, coarse_iters: int = 0, max_iters: int = 100,
                    tau: float = 1e-6, target: float = 0.0, check_every: int = 0, f=None, g=None,
                    online_iters: int = 0, lift_samples: int = 0, lift_tol: float = 0.0,
                    lift_rounds: int = 0, stream=None):
    """The block-sparse solver (see the C header for the method and its
    readings).  f, g are outputs (and inputs when coarse_iters == 0; zeros if
    None).  Returns (f, g, report) with report a dict of fs_sparse_report."""
    n, d = X.shape
    m = Y.shape[0]
    if f is None:
        f = _zeros_like(X, (n,))
    if g is None:
        g = _zeros_like(X, (m,))
    o = fs_sparse_options()
    o.coarse_iters, o.max_iters, o.check_every = int(coarse_iters), int(max_iters), int(check_every)
    o.tau, o.target = float(tau), float(target)
    o.online_iters = int(online_iters)
    o.lift_samples, o.lift_rounds, o.lift_tol = int(lift_samples), int(lift_rounds), float(lift_tol)
    rep = fs_sparse_report()
    st = load_library().fs_sparse_solve(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), ctypes.byref(o), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)), ctypes.byref(rep),
        _stream(stream, X, f))
    _raise(st)
    _host_sync(stream, f, g)
    return f, g, {k: getattr(rep, k) for k, _ in fs_sparse_report._fields_}


def _i_ptr(x, name: str, shape, dtype) -> int:
    import torch
    if not (_is_torch(x) and x.is_cuda and x.dtype == dtype and x.is_contiguous()
            and tuple(x.shape) == tuple(shape)):
        raise TypeError(f"{name} must be a contiguous CUDA {dtype} tensor of shape {tuple(shape)}")
    return x.data_ptr()


def fs_morton_order(X, Y, *, stream=None):
    """Morton order of both clouds (CUDA tensors): (perm_x, perm_y) int64."""
    import torch
    n, d = X.shape
    m = Y.shape[0]
    px = torch.empty(n, dtype=torch.int64, device=X.device)
    py = torch.empty(m, dtype=torch.int64, device=X.device)
    st = load_library().fs_morton_order(_ptr(X, "X", (n, d)), n, _ptr(Y, "Y", (m, d)), m, d,
                                        _i_ptr(px, "perm_x", (n,), torch.int64),
                                        _i_ptr(py, "perm_y", (m,), torch.int64), _stream(stream, X))
    _raise(st)
    return px, py


def fs_sparse_screen(X, a, Y, b, eps: float, f, g, tau: float, side: int, *, stream=None):
    """One screening at (f, g); side 0 for an f-update, 1 for a g-update.
    Returns (counts, lists) int32 CUDA tensors in Morton block numbering."""
    import torch
    n, d = X.shape
    m = Y.shape[0]
    nbx, nby = (n + 127) // 128, (m + 127) // 128
    no, ni = (nbx, nby) if side == 0 else (nby, nbx)
    counts = torch.empty(no, dtype=torch.int32, device=X.device)
    lists = torch.empty((no, ni), dtype=torch.int32, device=X.device)
    st = load_library().fs_sparse_screen(
        _ptr(X, "X", (n, d)), _ptr(a, "a", (n,)), n, _ptr(Y, "Y", (m, d)), _ptr(b, "b", (m,)), m, d,
        float(eps), _ptr(f, "f", (n,)), _ptr(g, "g", (m,)), float(tau), int(side),
        _i_ptr(counts, "counts", (no,), torch.int32), _i_ptr(lists, "lists", (no, ni), torch.int32),
        _stream(stream, X))
    _raise(st)
    return counts, lists


def fs_wait_selftest(timeout_ns: int = 1_000_000, *, stream=None) -> None:
    """Run the library's bounded device wait on a barrier nothing signals
    (see the C header); the next fs_check() raises FS_ERR_TIMEOUT."""
    _raise(load_library().fs_wait_selftest(int(timeout_ns), _stream(stream)))


def fs_barrier_selftest(timeout_ns: int = 1_000_000, *, stream=None) -> None:
    """Run the one-launch solve's grid barrier with a block that never
    arrives (see the C header); the next fs_check() raises FS_ERR_TIMEOUT."""
    _raise(load_library().fs_barrier_selftest(int(timeout_ns), _stream(stream)))
