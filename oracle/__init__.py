"""Float64 CPU oracle for the FlashSinkhorn hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never loads it, and this package never loads the product library: the two
share no code, header, table or helper.  Only the seeded input generators
(``streaming_sinkhorn_solver_gb300.workloads``, which hold none of the method's
arithmetic) feed both sides.

The arithmetic lives in ``sinkhorn_oracle.c`` (plain float64 C, OpenMP over
independent rows or columns).  This wrapper compiles it with gcc on first use
and exposes numpy-level functions.  Every function follows "FlashSinkhorn:
IO-Aware Entropic Optimal Transport on GPU" (gist.science technical summary):

* ``cost``              -- Problem statement: C_ij = ||x_i - y_j||^2.
* ``f_update`` / ``g_update`` / ``sinkhorn`` -- Method 1: the stabilised
  log-domain update f_i = -eps LSE_j[(g_j - C_ij)/eps + log b_j] and its
  symmetric g-update (reading: gamma_i = eps log a_i); one iteration is an
  f-update followed by a g-update from the new f.
* ``f_update_prop1``    -- Method 1, Proposition 1: the same f written as a row
  LSE of S_X = (Q K^T + 1(g_hat + delta)^T)/eps, Q = sqrt2 X, K = sqrt2 Y.
* ``apply_plan``, ``barycentric``, ``grad_x`` -- Method 3: plan application
  P V, the barycentric projection P Y / a and the gradient
  2(a_i x_i - (P Y)_i), with P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps).
* ``marginals``, ``transport_cost``, ``dual`` -- plan diagnostics.

Every function is pinned by ``tests/test_oracle.py`` against facts that do
not come from the oracle itself (closed forms, brute-force OT, invariances,
the Proposition 1 identity, finite differences).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sinkhorn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_P = np.ctypeslib.ndpointer
_f32 = _P(dtype=np.float32, flags="C_CONTIGUOUS")
_f64 = _P(dtype=np.float64, flags="C_CONTIGUOUS")
_i64 = _P(dtype=np.int64, flags="C_CONTIGUOUS")
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_DBL = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (float64, no fast-math, no FMA contraction)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_OUT_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    lib.orc_num_threads.restype = _INT
    lib.orc_set_num_threads.argtypes = [_INT]
    lib.orc_cost.argtypes = [_f32, _I64, _f32, _I64, _INT, _f64]
    lib.orc_cost_cosine.argtypes = [_f32, _I64, _f32, _I64, _INT, _f64]
    lib.orc_f_update.argtypes = [_f64, _I64, _I64, _f32, _DBL, _f64, _f64]
    lib.orc_g_update.argtypes = [_f64, _I64, _I64, _f32, _DBL, _f64, _f64]
    lib.orc_sinkhorn.argtypes = [_f64, _I64, _I64, _f32, _f32, _DBL, _INT, _f64, _f64]
    lib.orc_f_update_rows.argtypes = [_f32, _f32, _I64, _INT, _f32, _DBL, _f64, _i64, _I64, _f64]
    lib.orc_f_update_prop1.argtypes = [_f32, _I64, _f32, _I64, _INT, _f32, _DBL, _f64, _f64]
    lib.orc_apply_plan.argtypes = [_f64, _I64, _I64, _f32, _f32, _DBL, _f64, _f64, _f32, _INT, _f64]
    lib.orc_apply_plan_rows.argtypes = [_f32, _f32, _f32, _f32, _I64, _INT, _DBL, _f64, _f64,
                                        _f32, _INT, _i64, _I64, _f64]
    lib.orc_marginals.argtypes = [_f64, _I64, _I64, _f32, _f32, _DBL, _f64, _f64, _f64, _f64]
    lib.orc_transport_cost.argtypes = [_f64, _I64, _I64, _f32, _f32, _DBL, _f64, _f64]
    lib.orc_transport_cost.restype = _DBL
    _lib = lib
    return lib


class use_library:
    """Context manager: route every oracle call through another build of
    ``sinkhorn_oracle.c`` (the pin tests use it to load planted mutants)."""

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        _lib = None
        lib = ctypes.CDLL(self.path)
        ref = self.saved
        for name in dir(ref):
            if name.startswith("orc_"):
                fn, src = getattr(lib, name), getattr(ref, name)
                fn.argtypes = src.argtypes
                fn.restype = src.restype
        _lib = lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (same flags as build())."""
    c_path = out_path + ".c"
    with open(c_path, "w") as fh:
        fh.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                    "-ffp-contract=off", "-fno-fast-math", c_path, "-o", out_path, "-lm"],
                   check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as fh:
        return fh.read()


def _c32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _c64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(t: int) -> None:
    _load().orc_set_num_threads(int(t))


def as_eps(eps: float) -> float:
    """The regularisation both sides see: the float32 value, widened."""
    return float(np.float32(eps))


def cost(X, Y) -> np.ndarray:
    X, Y = _c32(X), _c32(Y)
    n, d = X.shape
    m = Y.shape[0]
    C = np.empty((n, m), dtype=np.float64)
    _load().orc_cost(X, n, Y, m, d, C)
    return C


def cost_cosine(X, Y) -> np.ndarray:
    """C_ij = 2 - 2 cos(x_i, y_j), from its definition (zero rows: see the C source)."""
    X, Y = _c32(X), _c32(Y)
    n, d = X.shape
    m = Y.shape[0]
    C = np.empty((n, m), dtype=np.float64)
    _load().orc_cost_cosine(X, n, Y, m, d, C)
    return C


def f_update(C, b, eps, g) -> np.ndarray:
    C = _c64(C)
    n, m = C.shape
    f = np.empty(n, dtype=np.float64)
    _load().orc_f_update(C, n, m, _c32(b), as_eps(eps), _c64(g), f)
    return f


def g_update(C, a, eps, f) -> np.ndarray:
    C = _c64(C)
    n, m = C.shape
    g = np.empty(m, dtype=np.float64)
    _load().orc_g_update(C, n, m, _c32(a), as_eps(eps), _c64(f), g)
    return g


def sinkhorn(C, a, b, eps, n_iter, f0=None, g0=None) -> Tuple[np.ndarray, np.ndarray]:
    """``n_iter`` iterations from (f0, g0) (zeros by default); returns (f, g)."""
    C = _c64(C)
    n, m = C.shape
    f = np.zeros(n) if f0 is None else _c64(f0).copy()
    g = np.zeros(m) if g0 is None else _c64(g0).copy()
    _load().orc_sinkhorn(C, n, m, _c32(a), _c32(b), as_eps(eps), int(n_iter), f, g)
    return f, g


def sinkhorn_stages(C, a, b, stages: Sequence[Tuple[float, int]], f0=None, g0=None):
    """Run (eps, iterations) stages back to back, each warm-started."""
    C = _c64(C)
    f = np.zeros(C.shape[0]) if f0 is None else _c64(f0)
    g = np.zeros(C.shape[1]) if g0 is None else _c64(g0)
    for eps, it in stages:
        f, g = sinkhorn(C, a, b, eps, it, f, g)
    return f, g


def f_update_rows(X, Y, b, eps, g, rows) -> np.ndarray:
    X, Y = _c32(X), _c32(Y)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    m, d = Y.shape
    out = np.empty(len(rows), dtype=np.float64)
    _load().orc_f_update_rows(X, Y, m, d, _c32(b), as_eps(eps), _c64(g), rows, len(rows), out)
    return out


def f_update_prop1(X, Y, b, eps, g) -> np.ndarray:
    X, Y = _c32(X), _c32(Y)
    n, d = X.shape
    m = Y.shape[0]
    f = np.empty(n, dtype=np.float64)
    _load().orc_f_update_prop1(X, n, Y, m, d, _c32(b), as_eps(eps), _c64(g), f)
    return f


def apply_plan(C, a, b, eps, f, g, V) -> np.ndarray:
    C = _c64(C)
    n, m = C.shape
    V = _c32(V)
    squeeze = V.ndim == 1
    V2 = V.reshape(m, -1)
    k = V2.shape[1]
    out = np.empty((n, k), dtype=np.float64)
    _load().orc_apply_plan(C, n, m, _c32(a), _c32(b), as_eps(eps), _c64(f), _c64(g),
                           np.ascontiguousarray(V2), k, out)
    return out[:, 0] if squeeze else out


def apply_plan_rows(X, a, Y, b, eps, f, g, V, rows) -> np.ndarray:
    X, Y, V = _c32(X), _c32(Y), _c32(V)
    m, d = Y.shape
    V2 = np.ascontiguousarray(V.reshape(m, -1))
    k = V2.shape[1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((len(rows), k), dtype=np.float64)
    _load().orc_apply_plan_rows(X, _c32(a), Y, _c32(b), m, d, as_eps(eps), _c64(f), _c64(g),
                                V2, k, rows, len(rows), out)
    return out


def barycentric(C, a, b, eps, f, g, Y) -> np.ndarray:
    """T_i = (P Y)_i / a_i (dividing by the weight a_i, not the realised row sum)."""
    out = apply_plan(C, a, b, eps, f, g, Y)
    return out / np.asarray(a, dtype=np.float64)[:, None]


def grad_x(C, X, a, b, eps, f, g, Y) -> np.ndarray:
    """grad_i = 2 (a_i x_i - (P Y)_i)."""
    PY = apply_plan(C, a, b, eps, f, g, Y)
    return 2.0 * (np.asarray(a, dtype=np.float64)[:, None] * np.asarray(X, dtype=np.float64) - PY)


def grad_x_cosine(C, X, a, b, eps, f, g, Y) -> np.ndarray:
    """Gradient with respect to the raw x_i under the cosine cost: the chain
    rule through x^_i = x_i / |x_i| applied to 2 (a_i x^_i - (P Y^)_i), i.e.
    J_i^T of it with J_i = (I - x^_i x^_i^T) / |x_i| (zero rows: 0)."""
    X = np.asarray(X, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    nx = np.linalg.norm(X, axis=1)
    ny = np.linalg.norm(Y, axis=1)
    Xh = np.where(nx[:, None] > 0, X / np.where(nx > 0, nx, 1.0)[:, None], 0.0)
    Yh = np.where(ny[:, None] > 0, Y / np.where(ny > 0, ny, 1.0)[:, None], 0.0)
    G = 2.0 * (np.asarray(a, dtype=np.float64)[:, None] * Xh
               - apply_plan(C, a, b, eps, f, g, Yh.astype(np.float32)))
    G = G - np.sum(Xh * G, axis=1, keepdims=True) * Xh
    return np.where(nx[:, None] > 0, G / np.where(nx > 0, nx, 1.0)[:, None], 0.0)


def hvp_x(C, X, a, b, eps, f, g, Y, V) -> np.ndarray:
    """Hessian of F(X) = <a, f*> + <b, g*> (the converged entropic OT value)
    applied to a direction V (n x d), derived here (the pages name a streaming
    HVP without a formula):

      grad_i = 2 (a_i x_i - sum_j P_ij y_j)                         (envelope)
      d/dt P_ij = P_ij (fdot_i + gdot_j - Cdot_ij) / eps,  Cdot_ij = 2 (x_i - y_j).v_i
      fixed point P 1 = a, P^T 1 = b, differentiated:
        a_i fdot_i + (P gdot)_i = sum_j P_ij Cdot_ij
        (P^T fdot)_j + b_j gdot_j = sum_i P_ij Cdot_ij
      (H V)_i = 2 a_i v_i - (2/eps) sum_j P_ij (fdot_i + gdot_j - Cdot_ij) y_j

    The system is singular along the gauge (fdot + t, gdot - t), which leaves
    (H V) unchanged; the minimum-norm least-squares solution is taken.  Dense
    float64 throughout (small problems only)."""
    C = _c64(C)
    n, m = C.shape
    X = np.asarray(X, np.float64)
    Y = np.asarray(Y, np.float64)
    V = np.asarray(V, np.float64)
    a64 = np.asarray(a, np.float64)
    b64 = np.asarray(b, np.float64)
    e = as_eps(eps)
    P = a64[:, None] * b64[None, :] * np.exp((np.asarray(f, np.float64)[:, None]
                                              + np.asarray(g, np.float64)[None, :] - C) / e)
    Cdot = 2.0 * (np.sum(X * V, axis=1)[:, None] - V @ Y.T)        # (x_i - y_j).v_i, doubled
    r = np.sum(P * Cdot, axis=1)
    c = np.sum(P * Cdot, axis=0)
    A = np.block([[np.diag(a64), P], [P.T, np.diag(b64)]])
    sol = np.linalg.lstsq(A, np.concatenate([r, c]), rcond=None)[0]
    fdot, gdot = sol[:n], sol[n:]
    W = P * (fdot[:, None] + gdot[None, :] - Cdot)
    return 2.0 * a64[:, None] * V - (2.0 / e) * (W @ Y)


def marginals(C, a, b, eps, f, g) -> Tuple[np.ndarray, np.ndarray]:
    C = _c64(C)
    n, m = C.shape
    row = np.empty(n)
    col = np.empty(m)
    _load().orc_marginals(C, n, m, _c32(a), _c32(b), as_eps(eps), _c64(f), _c64(g), row, col)
    return row, col


def transport_cost(C, a, b, eps, f, g) -> float:
    C = _c64(C)
    n, m = C.shape
    return float(_load().orc_transport_cost(C, n, m, _c32(a), _c32(b), as_eps(eps),
                                            _c64(f), _c64(g)))


def dual(a, b, f, g) -> float:
    """<a, f> + <b, g>."""
    return float(np.dot(np.asarray(a, np.float64), f) + np.dot(np.asarray(b, np.float64), g))
