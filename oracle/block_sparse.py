"""Float64 oracle of the block-sparse low-dimensional solver.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use
it, and it never loads the product library.

Source: the post "FlashSinkhorn 2: Block-Sparse Entropic Optimal Transport"
(patty.io).  The post describes the method in words only; each step below is
the plainest reading of its sections, written out in float64 numpy:

* *Coarse resolution first*: space is cut into cells, the problem is solved
  between the cells' centroids, and every point of a cell inherits its
  cell's potential ("the price learned by the centroid").
  Reading: the cells are the blocks of the Morton-sorted points (below); a
  cell's centroid is the weight-averaged point, its weight the sum of its
  points' weights; the centroid problem is the same log-domain Sinkhorn
  (the dense oracle) for a fixed number of iterations from zero.
* *How to cut space so that skipping is safe*: points are put in Morton
  (Z-order) so that a block of consecutive points is spatially compact, and
  a block pair of the plan is the interaction of two such groups.
  Reading: coordinates are quantised to 2^B cells per axis over the joint
  bounding box of both clouds (float32 arithmetic, as the kernels do), with
  B = min(21, floor(63 / d)) so that the interleaved code fits 64 bits (21
  for d <= 3; 15, 12, 10, 9 and 7 for d = 4 .. 8), the bits are interleaved
  (bit b of axis k at position b*d + k), points are sorted stably by that
  code, and cut into blocks of 128 consecutive points.
* *How to guarantee that skipping is safe*: every block's contribution is
  bounded, blocks below a threshold set by block mass are skipped, and the
  threshold bounds the error the skipped tiles can make in every row and
  every column.
  Reading (derived here): with block centroids c_I, c_J, Delta = c_I - c_J,
  u_i = x_i - c_I, v_j = y_j - c_J, the cost satisfies
      C_ij = |Delta + u_i - v_j|^2 >= |Delta|^2 + 2 Delta.u_i - 2 Delta.v_j,
  so the plan mass of the block pair is at most 2^U_IJ with
      U_IJ = log2 sum_{i in I} a_i 2^{(f_i - 2 Delta.u_i) L/eps}
           + log2 sum_{j in J} b_j 2^{(g_j + 2 Delta.v_j) L/eps}
           - |Delta|^2 L/eps,                              L = log2(e).
  (The linear terms cancel the potentials' variation inside matched blocks,
  which a plain box-distance bound would not.)  Before the f-update, row block
  I keeps column block J iff U_IJ + sigma_IJ >= log2(tau W_I / N_J), or J is
  the first maximiser of U_IJ over J; the omitted mass of row block I is then
  below tau W_I (W_I its weight, N_J the number of column blocks), i.e. the
  skipped tiles move the row marginal by at most tau in L1 for unit total
  mass.  The g-update screens columns the same way from the new f.  sigma_IJ
  = 1/16 + 2^-16 (|max_I psi| + |max_J chi| + |Delta|^2 L/eps) is a slack in
  favour of keeping, so the float32 evaluation on the GPU never omits a block
  the exact bound keeps.  tau = 0 keeps every block.
* *Can the lifted solution be trusted*: a sample of points is checked
  against its marginal; if the lifted potentials pass, the fine stage
  starts, else the centroid stage runs more iterations.
  Reading: the sample is ``lift_samples`` points of X evenly spaced in
  Morton order (position floor(s n / S)); the statistic is the mean over
  the sample of |(P 1)_i / a_i - 1| for the dense plan at the lifted (f, g),
  i.e. |2^{(f_i - f'_i) L/eps} - 1| with f'_i the dense f-update of point
  i (every column); the lift passes when it is at most ``lift_tol``, and
  otherwise another ``coarse_iters`` centroid iterations run from the
  centroid potentials reached, at most ``lift_rounds`` times.
* The kept blocks are then iterated: the f-update over the kept blocks of its
  row block, then the g-update over the kept blocks of its column block.  The
  row residual |P 1 - a|_1 of the block-sparse plan (measured with a fresh
  f-screening) is the stopping test, checked every ``check_every``
  iterations against ``target``.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

from . import as_eps, cost, f_update_rows, sinkhorn

MORTON_BITS = 21            # cells per axis 2^21 for d <= 3 (morton_bits for larger d)
BLOCK = 128
L2E = 1.4426950408889634074   # log2(e)


# ---------------------------------------------------------------------------
# Morton order

def morton_box(X, Y) -> Tuple[np.ndarray, np.ndarray]:
    """Per-axis min and max over both clouds (float32, exact)."""
    P = np.concatenate([np.asarray(X, np.float32), np.asarray(Y, np.float32)])
    return P.min(axis=0), P.max(axis=0)


def morton_bits(d: int) -> int:
    """Quantisation bits per axis: the d-axis code fits 64 bits."""
    return min(MORTON_BITS, 63 // d)


def morton_codes(P, lo, hi, bits: Optional[int] = None) -> np.ndarray:
    """Z-order codes: q_k = floor((p_k - lo_k) * (2^bits / (hi_k - lo_k))) in
    float32 arithmetic (each operation rounded once), clamped to
    [0, 2^bits - 1] (q = 0 on an axis of zero extent); bit b of q_k goes to
    bit b*d + k of the code.  bits defaults to morton_bits(d)."""
    P = np.asarray(P, np.float32)
    n, d = P.shape
    if bits is None:
        bits = morton_bits(d)
    lo = np.asarray(lo, np.float32)
    hi = np.asarray(hi, np.float32)
    span = (hi - lo).astype(np.float32)
    grid = np.float32(2 ** bits)
    with np.errstate(divide="ignore", invalid="ignore"):
        scale = np.where(span > 0, grid / np.where(span > 0, span, np.float32(1)),
                         np.float32(0)).astype(np.float32)
    t = (P - lo).astype(np.float32)
    u = (t * scale).astype(np.float32)
    q = np.clip(np.floor(u).astype(np.int64), 0, 2 ** bits - 1)
    codes = np.zeros(n, dtype=np.uint64)
    for b in range(bits):
        for k in range(d):
            bit = ((q[:, k] >> b) & 1).astype(np.uint64)
            codes |= bit << np.uint64(b * d + k)
    return codes


def morton_order(X, Y) -> Tuple[np.ndarray, np.ndarray]:
    """Stable sort of each cloud by its code (ties keep the input order)."""
    lo, hi = morton_box(X, Y)
    px = np.argsort(morton_codes(X, lo, hi), kind="stable")
    py = np.argsort(morton_codes(Y, lo, hi), kind="stable")
    return px.astype(np.int64), py.astype(np.int64)


# ---------------------------------------------------------------------------
# blocks and cells

def block_ids(count: int, block: int = BLOCK) -> np.ndarray:
    return np.arange(count) // block


def block_stats(Ps, ws, block: int = BLOCK) -> Tuple[np.ndarray, np.ndarray]:
    """Centroid and weight of each block of the sorted cloud ``Ps`` (weights
    ``ws``): W = sum of the weights and S = sum of w_i p_i, both accumulated in
    float64 in point order; centroid = float32(S / W), weight = float32(W)."""
    Ps = np.asarray(Ps, np.float32)
    ws = np.asarray(ws, np.float32)
    n, d = Ps.shape
    nb = (n + block - 1) // block
    W = np.zeros(nb)
    S = np.zeros((nb, d))
    for t in range(block):
        idx = np.arange(nb) * block + t
        ok = idx < n
        w = ws[idx[ok]].astype(np.float64)
        W[ok] = W[ok] + w
        S[ok] = S[ok] + w[:, None] * Ps[idx[ok]].astype(np.float64)
    return (S / W[:, None]).astype(np.float32), W.astype(np.float32)


def coarse_potentials(Xs, as_, Ys, bs, eps, iters, block: int = BLOCK, F0=None, G0=None):
    """Coarse stage: Sinkhorn between the block centroids (weights = block
    weights), from (F0, G0) (zeros by default), then every point inherits its
    block's potential.  Returns (f, g, (cx, wx, cy, wy), (F, G))."""
    cx, wx = block_stats(Xs, as_, block)
    cy, wy = block_stats(Ys, bs, block)
    F, G = sinkhorn(cost(cx, cy), wx, wy, eps, iters, F0, G0)
    return (F[block_ids(len(Xs), block)], G[block_ids(len(Ys), block)], (cx, wx, cy, wy),
            (F, G))


def lift_sample(n: int, samples: int) -> np.ndarray:
    """Positions (in Morton order) of the points the lift check samples."""
    s = min(int(samples), n)
    return (np.arange(s, dtype=np.int64) * n) // s


def lift_error(Xs, Ys, bs, eps, fs, gs, rows) -> float:
    """Mean over the sampled rows of |(P 1)_i / a_i - 1| for the dense plan
    at (fs, gs): (P 1)_i / a_i = exp((f_i - f'_i) / eps), f' the dense
    f-update (every column) from gs."""
    f_new = f_update_rows(Xs, Ys, bs, eps, gs, rows)
    r = np.exp((np.asarray(fs, np.float64)[rows] - f_new) / as_eps(eps))
    return float(np.mean(np.abs(r - 1.0)))


# ---------------------------------------------------------------------------
# screening

def block_bounds(Xs, as_, fs, Ys, bs, gs, eps, cx, cy, block: int = BLOCK):
    """U[I, J] (log2 of the bound on the plan mass of block pair (I, J)) and
    the slack sigma[I, J]."""
    e = as_eps(eps)
    Xs = np.asarray(Xs, np.float64)
    Ys = np.asarray(Ys, np.float64)
    cx = np.asarray(cx, np.float64)
    cy = np.asarray(cy, np.float64)
    psi = np.asarray(fs, np.float64) * (L2E / e) + np.log2(np.asarray(as_, np.float64))
    chi = np.asarray(gs, np.float64) * (L2E / e) + np.log2(np.asarray(bs, np.float64))
    kap = 2.0 * L2E / e
    nI, nJ = len(cx), len(cy)
    bj = block_ids(len(Ys), block)
    starts = np.arange(nJ) * block
    v = Ys - cy[bj]                                   # v_j = y_j - c_J(j)
    chi_max = np.maximum.reduceat(chi, starts)
    U = np.empty((nI, nJ))
    sig = np.empty((nI, nJ))
    for I in range(nI):
        ri = slice(I * block, min((I + 1) * block, len(Xs)))
        u = Xs[ri] - cx[I]                            # u_i = x_i - c_I
        D = cx[I][None, :] - cy                       # Delta for every J
        Z = psi[ri][:, None] - kap * (u @ D.T)        # |I| x nJ
        zm = Z.max(axis=0)
        A = zm + np.log2(np.sum(np.exp2(Z - zm[None, :]), axis=0))
        W = chi + kap * np.sum(v * D[bj], axis=1)     # m
        wm = np.maximum.reduceat(W, starts)
        B = wm + np.log2(np.add.reduceat(np.exp2(W - wm[bj]), starts))
        dd = np.sum(D * D, axis=1) * (L2E / e)
        U[I] = A + B - dd
        sig[I] = 1.0 / 16 + 2.0 ** -16 * (abs(psi[ri].max()) + np.abs(chi_max) + dd)
    return U, sig


def screen(U, sig, w_out, tau: float, side: str) -> np.ndarray:
    """Kept-block mask [output blocks x input blocks].  side 'x': rows of U
    are the output (f-update); side 'y': columns are (g-update)."""
    if side == "y":
        U, sig = U.T, sig.T
    nO, nIn = U.shape
    if tau <= 0:
        return np.ones((nO, nIn), dtype=bool)
    T = np.log2(np.float64(tau)) + np.log2(np.asarray(w_out, np.float64)) - np.log2(nIn)
    keep = U + sig >= T[:, None]
    keep[np.arange(nO), np.argmax(U, axis=1)] = True
    return keep


def omitted_mass(C, as_, bs, eps, fs, gs, keep_x, block: int = BLOCK) -> np.ndarray:
    """Plan mass of the omitted block pairs per row block (brute force)."""
    e = as_eps(eps)
    P = (np.asarray(as_, np.float64)[:, None] * np.asarray(bs, np.float64)[None, :]
         * np.exp((np.asarray(fs)[:, None] + np.asarray(gs)[None, :] - C) / e))
    bi = block_ids(C.shape[0], block)
    bj = block_ids(C.shape[1], block)
    mask = keep_x[bi][:, bj]
    out = np.zeros(keep_x.shape[0])
    np.add.at(out, bi, np.where(mask, 0.0, P).sum(axis=1))
    return out


# ---------------------------------------------------------------------------
# the block-sparse iteration

def _masked_lse(Z: np.ndarray, mask: np.ndarray) -> np.ndarray:
    Z = np.where(mask, Z, -np.inf)
    mx = Z.max(axis=1)
    return mx + np.log(np.sum(np.exp(Z - mx[:, None]), axis=1))


def sparse_f_update(C, bs, eps, gs, keep_x, block: int = BLOCK) -> np.ndarray:
    """f_i = -eps LSE over the kept columns of (g_j - C_ij)/eps + log b_j."""
    e = as_eps(eps)
    mask = keep_x[block_ids(C.shape[0], block)][:, block_ids(C.shape[1], block)]
    Z = (np.asarray(gs, np.float64)[None, :] - C) / e + np.log(np.asarray(bs, np.float64))[None, :]
    return -e * _masked_lse(Z, mask)


def sparse_g_update(C, as_, eps, fs, keep_y, block: int = BLOCK) -> np.ndarray:
    """g_j = -eps LSE over the kept rows of (f_i - C_ij)/eps + log a_i."""
    e = as_eps(eps)
    mask = keep_y[block_ids(C.shape[1], block)][:, block_ids(C.shape[0], block)]
    Z = (np.asarray(fs, np.float64)[None, :] - C.T) / e + np.log(np.asarray(as_, np.float64))[None, :]
    return -e * _masked_lse(Z, mask)


def row_residual(C, as_, bs, eps, fs, gs, keep_x, block: int = BLOCK) -> float:
    """|P 1 - a|_1 of the block-sparse plan (kept blocks of the f-screening)."""
    e = as_eps(eps)
    mask = keep_x[block_ids(C.shape[0], block)][:, block_ids(C.shape[1], block)]
    P = (np.asarray(as_, np.float64)[:, None] * np.asarray(bs, np.float64)[None, :]
         * np.exp((np.asarray(fs)[:, None] + np.asarray(gs)[None, :] - C) / e))
    r = np.where(mask, P, 0.0).sum(axis=1)
    return float(np.abs(r - np.asarray(as_, np.float64)).sum())


def solve(X, a, Y, b, eps, coarse_iters: int, max_iters: int, tau: float,
          target: float = 0.0, check_every: int = 0, f0=None, g0=None,
          block: int = BLOCK, lift_samples: int = 0, lift_tol: float = 0.0,
          lift_rounds: int = 0) -> Tuple[np.ndarray, np.ndarray, Dict]:
    """The whole solver: Morton order, coarse stage (or the caller's f0, g0
    when coarse_iters == 0) with the lift check (lift_samples > 0), block-
    sparse iterations with the stopping test, and the final residual.
    Returns (f, g, report) in the caller's order."""
    X = np.asarray(X, np.float32)
    Y = np.asarray(Y, np.float32)
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    px, py = morton_order(X, Y)
    Xs, as_, Ys, bs = X[px], a[px], Y[py], b[py]
    cx, wx = block_stats(Xs, as_, block)
    cy, wy = block_stats(Ys, bs, block)
    lift_checks, lift_err = 0, -1.0
    if coarse_iters > 0:
        fs, gs, _, (F, G) = coarse_potentials(Xs, as_, Ys, bs, eps, coarse_iters, block)
        if lift_samples > 0:
            rows = lift_sample(len(Xs), lift_samples)
            lift_err = lift_error(Xs, Ys, bs, eps, fs, gs, rows)
            lift_checks = 1
            while lift_err > lift_tol and lift_checks <= lift_rounds:
                fs, gs, _, (F, G) = coarse_potentials(Xs, as_, Ys, bs, eps, coarse_iters, block,
                                                      F, G)
                lift_err = lift_error(Xs, Ys, bs, eps, fs, gs, rows)
                lift_checks += 1
    else:
        fs = np.zeros(len(X)) if f0 is None else np.asarray(f0, np.float64)[px]
        gs = np.zeros(len(Y)) if g0 is None else np.asarray(g0, np.float64)[py]
    C = cost(Xs, Ys)
    nI, nJ = len(cx), len(cy)
    rep = {"iters": 0, "kept_blocks": 0, "kept_pairs": 0, "halves": 0,
           "blocks_x": nI, "blocks_y": nJ, "lift_checks": lift_checks, "lift_error": lift_err}
    sx = np.minimum(block, len(X) - np.arange(nI) * block)
    sy = np.minimum(block, len(Y) - np.arange(nJ) * block)

    def screen_x():
        U, sig = block_bounds(Xs, as_, fs, Ys, bs, gs, eps, cx, cy, block)
        return screen(U, sig, wx, tau, "x")

    it = 0
    while it < max_iters:
        if target > 0 and check_every > 0 and it > 0 and it % check_every == 0:
            if row_residual(C, as_, bs, eps, fs, gs, screen_x(), block) <= target:
                break
        kx = screen_x()
        fs = sparse_f_update(C, bs, eps, gs, kx, block)
        U, sig = block_bounds(Xs, as_, fs, Ys, bs, gs, eps, cx, cy, block)
        ky = screen(U, sig, wy, tau, "y")
        gs = sparse_g_update(C, as_, eps, fs, ky, block)
        rep["kept_blocks"] += int(kx.sum() + ky.sum())
        rep["kept_pairs"] += int((kx * sx[:, None] * sy[None, :]).sum()
                                 + (ky * sy[:, None] * sx[None, :]).sum())
        rep["halves"] += 2
        it += 1
    rep["iters"] = it
    rep["residual"] = row_residual(C, as_, bs, eps, fs, gs, screen_x(), block)
    f = np.empty(len(X))
    g = np.empty(len(Y))
    f[px] = fs
    g[py] = gs
    return f, g, rep
