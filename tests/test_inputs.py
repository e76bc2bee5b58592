"""Seeded workload generators: determinism and the structure each config states."""
import numpy as np
import pytest

from gated_deltanet_verification_gb300 import inputs as I


def _depths(parent):
    d = np.zeros(len(parent), np.int64)
    for i, p in enumerate(parent):
        d[i] = 0 if p < 0 else d[p] + 1
    return d


def test_deterministic():
    a, b = I.config_batch(1), I.config_batch(1)
    for f in ("parent", "q", "k", "v", "gamma", "beta", "S_pre", "accepted"):
        assert np.array_equal(getattr(a, f), getattr(b, f))


@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_random_tree_configs(cfg):
    b = I.config_batch(cfg)
    D = {0: 3, 1: 6, 2: 8}[cfg]
    sizes = b.tree_sizes()
    assert np.all(sizes == {0: 8, 1: 32, 2: 32}[cfg])
    for r in range(b.B):
        par = b.parent[b.offsets[r]:b.offsets[r + 1]]
        assert par[0] == -1 and np.all(par[1:] >= 0)  # single root child
        assert all(p < i for i, p in enumerate(par))
        assert _depths(par).max() <= D
    # L2-normalised q, k; gates in range
    nq = np.linalg.norm(b.q.astype(np.float64), axis=-1)
    assert np.allclose(nq, 1.0, atol=1e-2 if b.dtype == "bf16" else 1e-6)
    assert np.all((b.gamma > 0) & (b.gamma < 1)) and np.all((b.beta > 0) & (b.beta < 1))
    if b.dtype == "bf16":
        assert np.array_equal(I.round_to_bf16(b.q), b.q)


def test_budgeted_forest_config():
    b = I.config_batch(3)
    sizes = b.tree_sizes()
    assert b.B == 64 and b.N <= 2048 and sizes.min() >= 1 and sizes.max() <= 64
    for r in range(b.B):
        par = b.parent[b.offsets[r]:b.offsets[r + 1]]
        assert all(p < i for i, p in enumerate(par))
        assert _depths(par).max() <= 12
        # every node has at most 4 children
        kids = np.bincount(par[par >= 0], minlength=len(par))
        assert kids.max(initial=0) <= 4
        assert np.sum(par == -1) <= 4


@pytest.mark.parametrize("shape,depth,acc", [("chain", 127, 127), ("star", 0, 0), ("4ary", 3, 84)])
def test_shape_extremes(shape, depth, acc):
    b = I.config_batch(4, shape=shape)
    assert b.B == 8 and b.N == 1024
    par = b.parent[:128]
    assert _depths(par).max() == depth
    assert np.all(b.accepted == acc)


def test_bf16_rounding_matches_ties_to_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even mantissa (1.0)
    y = I.round_to_bf16(x)
    assert y[0] == 1.0 and y[1] == 1.0 and y[2] == np.float32(1.015625)
    assert y[3] == -2.5
