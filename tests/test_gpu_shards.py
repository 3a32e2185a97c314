"""Row-sharded half-updates on one GPU (fs_options.row_shards).

Every half-update runs as G shards of whole row blocks of the updated side,
the launches a G-GPU row partition would make, one after the other; each
launch sees only its rows.  The solve must equal the one-launch solve bit
for bit (same column split, same per-row arithmetic) on the FMA path, the
one-CTA tensor path and the CTA-pair tensor path, with online maxima and
with reference offsets and fixups, for ragged sizes, uneven shards and more
shards than row blocks."""
import numpy as np
import pytest

from streaming_sinkhorn_solver_gb300 import binding as fs
from streaming_sinkhorn_solver_gb300.workloads import make_inputs, random_cloud
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    fs.load_library()


def _inputs(kind):
    if kind == "fma_ref":          # n m = 7.4e7 > 2^26: reference offsets from iteration 3
        return make_inputs("c2_n10k_d3", n=9000, m=8200, seed=301), 0.005, 6, "fma"
    if kind == "fma_fold":         # n m = 2.7e8 >= 2^28: Morton order, offsets folded per CTA
        return make_inputs("c2_n10k_d3", n=16400, m=16400, seed=306), 0.01, 5, "fma"
    if kind == "fma_small":        # online maxima only
        return random_cloud(1500, 1000, 8, seed=302, spread=0.5, weights="lognormal"), 0.05, 4, "fma"
    if kind == "tc_ref":           # one-CTA tensor kernels, reference offsets
        return make_inputs("c3_n50k_d64", n=8300, m=8200, seed=303), 0.1, 5, "tensor"
    if kind == "pair_ref":         # CTA-pair kernels (d > 128), reference offsets
        return random_cloud(8300, 8200, 200, seed=304, spread=200 ** -0.5,
                            weights="lognormal"), 0.5, 5, "tensor"
    if kind == "tc_small":         # ragged, online maxima only
        return random_cloud(700, 900, 48, seed=305, spread=48 ** -0.5), 0.1, 3, "tensor"
    raise KeyError(kind)


def _solve(t, eps, iters, path, splits, shards):
    f, g = fs.fs_sinkhorn_solve(t["X"], t["a"], t["Y"], t["b"], eps, iters, path=path,
                                splits=splits, row_shards=shards)
    return f.cpu().numpy(), g.cpu().numpy()


@pytest.mark.parametrize("kind", ["fma_ref", "fma_fold", "fma_small", "tc_ref", "pair_ref",
                                  "tc_small"])
@pytest.mark.parametrize("splits", [0, 1])
def test_row_shards_are_bitwise_the_unsharded_solve(kind, splits):
    import torch
    inp, eps, iters, path = _inputs(kind)
    t = to_dev(inp)
    n, d = inp["X"].shape
    m = inp["Y"].shape[0]
    unit = fs.fs_shard_unit(d, path)
    f1, g1 = _solve(t, eps, iters, path, splits, 0)
    assert np.isfinite(f1).all() and np.isfinite(g1).all()
    units = max(-(-n // unit), -(-m // unit))
    for shards in (2, 3, units + 3):
        torch.cuda.synchronize()
        before = fs.fs_launch_count()
        fG, gG = _solve(t, eps, iters, path, splits, shards)
        launched = fs.fs_launch_count() - before
        assert fG.tobytes() == f1.tobytes(), (kind, splits, shards)
        assert gG.tobytes() == g1.tobytes(), (kind, splits, shards)
        # one half-update launch per non-empty shard and half
        nonempty_f = sum(1 for s in range(shards) if np.diff(fs.fs_shard_range(n, unit, shards, s))[0] > 0)
        nonempty_g = sum(1 for s in range(shards) if np.diff(fs.fs_shard_range(m, unit, shards, s))[0] > 0)
        assert launched >= iters * (nonempty_f + nonempty_g)


def test_row_shards_with_host_buffers():
    inp, eps, iters, path = _inputs("fma_small")
    t = to_dev(inp)
    f1, g1 = _solve(t, eps, iters, path, 0, 0)
    fh, gh = fs.fs_sinkhorn_solve(inp["X"], inp["a"], inp["Y"], inp["b"], eps, iters, path=path,
                                  row_shards=4)
    assert fh.tobytes() == f1.tobytes() and gh.tobytes() == g1.tobytes()
