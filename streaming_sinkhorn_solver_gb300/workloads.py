"""Seeded synthetic point-cloud workloads.

This module only draws inputs.  It holds none of the solver's arithmetic, so
both the CUDA path and the float64 oracle can consume the same arrays without
sharing any code of the method.

The FlashSinkhorn pages ("FlashSinkhorn: IO-Aware Entropic Optimal Transport on
GPU", Experimental results) evaluate on synthetic point clouds up to n = 50,000
and d = 1024 without stating their distributions.  The five workloads below
stand in for them; each is a fixed recipe of shapes, distributions, weights,
regularisation schedule and the plan operator applied afterwards.

All arrays are drawn in float64 with ``numpy.random.default_rng(seed)`` and
cast to float32, row-major and contiguous.  Weights are normalised to sum 1 in
float64 before the cast; neither side renormalises them afterwards.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional, Tuple

import numpy as np

__all__ = ["Workload", "WORKLOADS", "make_inputs", "eps_schedule", "random_cloud", "clustered_cloud"]


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    m: int
    d: int
    # (eps, iterations) stages; a plain solve has one stage.
    stages: Tuple[Tuple[float, int], ...]
    # plan operator applied after the solve: None, "barycentric", "grad_x" or "pv"
    apply: Optional[str]
    k: int = 0          # columns of V for "pv"
    seed: int = 0
    about: str = ""
    # block-sparse solver only: coarse centroid iterations and the screening's
    # omitted-mass bound (0 = the dense solver)
    coarse_iters: int = 0
    tau: float = 0.0

    @property
    def n_iter(self) -> int:
        return sum(it for _, it in self.stages)


def eps_schedule(eps_start: float, eps_end: float, n_stages: int, iters: int):
    """Geometric schedule with both end points included."""
    if n_stages == 1:
        return ((float(eps_end), iters),)
    r = (eps_end / eps_start) ** (1.0 / (n_stages - 1))
    return tuple((float(eps_start * r ** s), iters) for s in range(n_stages))


WORKLOADS: Dict[str, Workload] = {
    "c1_n512_d2": Workload(
        "c1_n512_d2", 512, 512, 2, ((0.05, 100),), None, seed=1001,
        about="X~N(0,I), Y~N((1,1),0.5^2 I), uniform weights, eps=0.05, 100 iterations"),
    "c2_n10k_d3": Workload(
        "c2_n10k_d3", 10_000, 10_000, 3, ((0.01, 200),), "barycentric", seed=1002,
        about="X~U[0,1]^3, Y 4-component isotropic GMM (sigma 0.1), uniform weights, "
              "eps=0.01, 200 iterations, barycentric projection P.Y/a"),
    # The n=m=50,000, d=3 point of the throughput metric: the 10k recipe above
    # (same distributions, eps and plan operator) at the 50k size.
    "c2_n50k_d3": Workload(
        "c2_n50k_d3", 50_000, 50_000, 3, ((0.01, 100),), "barycentric", seed=1006,
        about="X~U[0,1]^3, Y 4-component isotropic GMM (sigma 0.1), uniform weights, "
              "eps=0.01, 100 iterations at n=m=50k, barycentric projection P.Y/a"),
    "c3_n50k_d64": Workload(
        "c3_n50k_d64", 50_000, 50_000, 64, ((0.1, 100),), None, seed=1003,
        about="X,Y~N(0,I/d), Y shifted 0.5 along e1, Dirichlet(1) weights, eps=0.1, "
              "100 iterations, forward only"),
    "c4_n50k_d512": Workload(
        "c4_n50k_d512", 50_000, 50_000, 512, ((0.05, 100),), "grad_x", seed=1004,
        about="X,Y rows N(0,I) scaled to unit norm, uniform weights, eps=0.05, "
              "100 iterations, then grad_x = 2(a x - P Y)"),
    "c5_n20k_m30k_d1024": Workload(
        "c5_n20k_m30k_d1024", 20_000, 30_000, 1024, eps_schedule(1.0, 0.01, 10, 20), "pv",
        k=64, seed=1005,
        about="X~N(0,I/d), Y~N(0,2I/d), log-normal weights, eps 1.0->0.01 geometric over "
              "10 stages x 20 iterations, final P.V with V~N(0,1) of shape m x 64"),
    "bs_n1m_d3": Workload(
        "bs_n1m_d3", 1_000_000, 1_000_000, 3, ((0.001, 50),), None, seed=1007,
        coarse_iters=50, tau=1e-6,
        about="block-sparse solver: the c2 recipe (X~U[0,1]^3, Y 4-component GMM sigma 0.1, "
              "uniform weights) at n=m=1e6, eps=1e-3 (blur 0.03, three mean spacings), 50 "
              "centroid iterations, then 50 block-sparse iterations with tau=1e-6"),
    # the same recipe at four times the points, eps scaled with the squared mean
    # spacing (4^(2/3)) so that a point still interacts with as many neighbours
    "bs_n4m_d3": Workload(
        "bs_n4m_d3", 4_000_000, 4_000_000, 3, ((0.00036, 20),), None, seed=1008,
        coarse_iters=50, tau=1e-6,
        about="block-sparse solver at n=m=4e6: the c2 recipe, eps=3.6e-4 (blur 0.019, three "
              "mean spacings), 50 centroid iterations, then 20 block-sparse iterations with "
              "tau=1e-6"),
    # sixteen times the points of bs_n1m_d3 (125,000^2 block pairs: the kept lists
    # no longer fit one row of every block per output block)
    "bs_n16m_d3": Workload(
        "bs_n16m_d3", 16_000_000, 16_000_000, 3, ((0.000142, 20),), None, seed=1009,
        coarse_iters=50, tau=1e-6,
        about="block-sparse solver at n=m=1.6e7: the c2 recipe, eps=1.42e-4 (blur 0.012, three "
              "mean spacings), 50 centroid iterations, then 20 block-sparse iterations with "
              "tau=1e-6"),
}


def _normalise(w: np.ndarray) -> np.ndarray:
    return (w / w.sum()).astype(np.float32)


def make_inputs(name: str, n: Optional[int] = None, m: Optional[int] = None,
                d: Optional[int] = None, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Draw the arrays of workload ``name``, optionally at a reduced size.

    Returns float32 arrays ``X`` (n x d), ``Y`` (m x d), ``a`` (n), ``b`` (m)
    and, for the "pv" workload, ``V`` (m x k).  A reduced size keeps every
    distribution of the recipe; only the counts change.
    """
    w = WORKLOADS[name]
    n = w.n if n is None else int(n)
    m = w.m if m is None else int(m)
    d = w.d if d is None else int(d)
    rng = np.random.default_rng(w.seed if seed is None else seed)
    out: Dict[str, np.ndarray] = {}
    if name.startswith("c1"):
        X = rng.standard_normal((n, d))
        Y = 1.0 + 0.5 * rng.standard_normal((m, d))
        a = np.full(n, 1.0 / n)
        b = np.full(m, 1.0 / m)
    elif name.startswith("c2") or name.startswith("bs"):
        X = rng.uniform(0.0, 1.0, (n, d))
        means = rng.uniform(0.0, 1.0, (4, d))
        comp = rng.integers(0, 4, m)
        Y = means[comp] + 0.1 * rng.standard_normal((m, d))
        a = np.full(n, 1.0 / n)
        b = np.full(m, 1.0 / m)
    elif name.startswith("c3"):
        X = rng.standard_normal((n, d)) / np.sqrt(d)
        Y = rng.standard_normal((m, d)) / np.sqrt(d)
        Y[:, 0] += 0.5
        a = rng.dirichlet(np.ones(n)) if n > 1 else np.ones(1)
        b = rng.dirichlet(np.ones(m)) if m > 1 else np.ones(1)
    elif name.startswith("c4"):
        X = rng.standard_normal((n, d))
        Y = rng.standard_normal((m, d))
        X /= np.linalg.norm(X, axis=1, keepdims=True)
        Y /= np.linalg.norm(Y, axis=1, keepdims=True)
        a = np.full(n, 1.0 / n)
        b = np.full(m, 1.0 / m)
    elif name.startswith("c5"):
        X = rng.standard_normal((n, d)) / np.sqrt(d)
        Y = rng.standard_normal((m, d)) * np.sqrt(2.0 / d)
        a = np.exp(rng.standard_normal(n))
        b = np.exp(rng.standard_normal(m))
        out["V"] = np.ascontiguousarray(rng.standard_normal((m, w.k)).astype(np.float32))
    else:  # pragma: no cover
        raise KeyError(name)
    out["X"] = np.ascontiguousarray(X.astype(np.float32))
    out["Y"] = np.ascontiguousarray(Y.astype(np.float32))
    out["a"] = _normalise(np.asarray(a, dtype=np.float64))
    out["b"] = _normalise(np.asarray(b, dtype=np.float64))
    return out


def random_cloud(n: int, m: int, d: int, seed: int, spread: float = 1.0,
                 shift: float = 0.0, weights: str = "uniform") -> Dict[str, np.ndarray]:
    """Generic Gaussian clouds for ragged-shape and edge-case tests."""
    rng = np.random.default_rng(seed)
    X = spread * rng.standard_normal((n, d)) + shift
    Y = spread * rng.standard_normal((m, d)) + shift + 0.25
    if weights == "uniform":
        a = np.full(n, 1.0 / n)
        b = np.full(m, 1.0 / m)
    else:
        a = np.exp(rng.standard_normal(n))
        b = np.exp(rng.standard_normal(m))
    return {"X": np.ascontiguousarray(X.astype(np.float32)),
            "Y": np.ascontiguousarray(Y.astype(np.float32)),
            "a": _normalise(a), "b": _normalise(b)}


def clustered_cloud(n: int, m: int, d: int, k: int, sigma: float, seed: int) -> Dict[str, np.ndarray]:
    """Both clouds drawn from one mixture of k isotropic Gaussians (standard
    deviation sigma) with means uniform in [0, 1]^d, uniform weights: points
    of low intrinsic extent in d = 4..8 dimensions, where block screening has
    whole cluster pairs to skip."""
    rng = np.random.default_rng(seed)
    means = rng.uniform(0.0, 1.0, (k, d))
    X = means[rng.integers(0, k, n)] + sigma * rng.standard_normal((n, d))
    Y = means[rng.integers(0, k, m)] + sigma * rng.standard_normal((m, d))
    return {"X": np.ascontiguousarray(X.astype(np.float32)),
            "Y": np.ascontiguousarray(Y.astype(np.float32)),
            "a": _normalise(np.full(n, 1.0 / n)), "b": _normalise(np.full(m, 1.0 / m))}
