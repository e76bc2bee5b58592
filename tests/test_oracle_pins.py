"""Pins for the CPU oracle: each check comes from the pages' mathematics or a
hand derivation, never from the oracle itself.  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle
from conftest import make_tree_batch, rel_fro
from gated_deltanet_verification_gb300 import inputs as I
from pins_lib import (all_parent_arrays, ancestors_or_self, closed_form_batch, closed_form_unit,
                      commit_from_factors, token_order_gdn, unit_factors)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_batch():
    with open(os.path.join(GOLDEN, "worked_tree3.json")) as f:
        g = json.load(f)
    b = make_tree_batch([g["parent"]], g["S_pre"], g["q"], g["k"], g["v"], g["gamma"], g["beta"])
    return g, b


def test_golden_worked_example():
    g, b = _golden_batch()
    O, U, logP = oracle.verify(b, nthreads=1)
    exp = g["expected"]
    np.testing.assert_allclose(U[:, 0], np.array(exp["u"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(O[:, 0], np.array(exp["o"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(np.exp(logP[:, 0]), np.array(exp["P"]), rtol=1e-15)
    depth, anc, req, st = oracle.pack(b.offsets, b.parent, 5)
    assert st == oracle.OK
    assert depth.tolist() == exp["depth"]
    for a_str, S_exp in exp["S_commit"].items():
        S_new = oracle.commit(b, accepted=np.array([int(a_str)], np.int32), nthreads=1)
        np.testing.assert_allclose(S_new[0, 0], np.array(S_exp), rtol=0, atol=1e-15)


def _random_unit_batch(rng, parent, dk=3, dv=5, H=1, dtype="f32"):
    T = len(parent)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    gamma = np.exp(-np.logaddexp(0, rng.standard_normal((T, H))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    S = rng.standard_normal((1, H, dk, dv)) * 0.3
    return make_tree_batch([parent], S, q, k, v, gamma, beta)


def test_closed_form_exhaustive_small_trees():
    """Theorem 1 with a dense solve equals sequential execution on every tree
    shape with up to 5 nodes (1 + 1 + 2 + 6 + 24 + 120 shapes)."""
    rng = np.random.default_rng(7)
    count = 0
    for T in range(1, 6):
        for parent in all_parent_arrays(T):
            b = _random_unit_batch(rng, parent)
            O, U, logP = oracle.verify(b, nthreads=1)
            Oc, Uc, logPc = closed_form_batch(b)
            assert rel_fro(O, Oc) < 1e-12, parent
            assert rel_fro(U, Uc) < 1e-12, parent
            np.testing.assert_allclose(logP, logPc, rtol=1e-13, atol=1e-14)
            count += 1
    assert count == 1 + 2 + 6 + 24 + 120


@pytest.mark.parametrize("seed", range(6))
def test_closed_form_random_trees(seed):
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(6, 17))
    parent = I.random_parent_tree(rng, T, int(rng.integers(1, T)))
    b = _random_unit_batch(rng, parent, dk=4, dv=6, H=2)
    O, U, logP = oracle.verify(b, nthreads=2)
    Oc, Uc, logPc = closed_form_batch(b)
    assert rel_fro(O, Oc) < 1e-12
    assert rel_fro(U, Uc) < 1e-12
    np.testing.assert_allclose(logP, logPc, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("shape", ["random", "chain", "4ary"])
def test_nilpotency_and_neumann(shape):
    """Lemma 3: G^(d+1) is exactly zero, G^d is not, and the finite Neumann
    sum equals the inverse of I + G."""
    rng = np.random.default_rng(11)
    T = 12
    if shape == "random":
        parent = I.random_parent_tree(rng, T, 4)
    elif shape == "chain":
        parent = I.chain_tree(T)
    else:
        parent = I.kary_tree(T)
    anc = ancestors_or_self(parent)
    d = max(len(s) for s in anc) - 1
    q = rng.standard_normal((T, 5))
    k = rng.standard_normal((T, 5))
    gamma = rng.uniform(0.3, 0.99, T)
    beta = rng.uniform(0.1, 0.9, T)
    _, G, _ = unit_factors(parent, q, k, gamma, beta)
    assert np.all(np.triu(G) == 0.0)  # strictly lower triangular
    Gd = np.linalg.matrix_power(G, d)
    Gd1 = Gd @ G
    assert np.all(Gd1 == 0.0)
    assert d == 0 or np.any(Gd != 0.0)
    neu = sum(np.linalg.matrix_power(-G, m) for m in range(d + 1))
    np.testing.assert_allclose(neu, np.linalg.inv(np.eye(T) + G), rtol=1e-12, atol=1e-14)
    assert abs(np.linalg.det(np.eye(T) + G) - 1.0) < 1e-12


def test_chain_reduces_to_token_order_gdn():
    rng = np.random.default_rng(3)
    T, dk, dv = 20, 6, 7
    b = _random_unit_batch(rng, I.chain_tree(T), dk, dv)
    O, U, _ = oracle.verify(b, nthreads=1)
    Ot, Ut, St = token_order_gdn(b.S_pre[0, 0], b.q[:, 0], b.k[:, 0], b.v[:, 0],
                                 b.gamma[:, 0].astype(np.float64), b.beta[:, 0].astype(np.float64))
    assert rel_fro(O[:, 0], Ot) < 1e-13
    assert rel_fro(U[:, 0], Ut) < 1e-13
    S_new = oracle.commit(b, accepted=np.array([T - 1], np.int32), nthreads=1)
    assert rel_fro(S_new[0, 0], St) < 1e-13


def test_star_gives_local_deltas():
    """All nodes are root children (d = 0): U equals the local deltas R and
    O_i = gamma_i S_pre^T q_i + (q_i.k_i) u_i."""
    rng = np.random.default_rng(5)
    T, dk, dv = 9, 4, 3
    b = _random_unit_batch(rng, I.star_tree(T), dk, dv)
    O, U, _ = oracle.verify(b, nthreads=1)
    S0 = b.S_pre[0, 0].astype(np.float64)
    for i in range(T):
        g, bt = float(b.gamma[i, 0]), float(b.beta[i, 0])
        qi, ki, vi = (x[i, 0].astype(np.float64) for x in (b.q, b.k, b.v))
        r = bt * (vi - g * S0.T @ ki)
        np.testing.assert_allclose(U[i, 0], r, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(O[i, 0], g * S0.T @ qi + (qi @ ki) * r, rtol=1e-12, atol=1e-15)


def test_zero_write_gate():
    """beta = 0: nothing is written, U = 0 and O = D_P Q S_pre."""
    rng = np.random.default_rng(9)
    b = _random_unit_batch(rng, I.random_parent_tree(rng, 10, 3), 4, 5)
    b.beta[:] = 0.0
    O, U, logP = oracle.verify(b, nthreads=1)
    assert np.all(U == 0.0)
    P = np.exp(logP[:, 0])
    expected = P[:, None] * (b.q[:, 0].astype(np.float64) @ b.S_pre[0, 0].astype(np.float64))
    np.testing.assert_allclose(O[:, 0], expected, rtol=1e-12, atol=1e-15)


def test_sibling_relabelling_invariance():
    """Renumbering the nodes in another parent-before-child order permutes the outputs."""
    rng = np.random.default_rng(21)
    T = 14
    parent = I.random_parent_tree(rng, T, 5)
    b = _random_unit_batch(rng, parent, 4, 4)
    O, U, logP = oracle.verify(b, nthreads=1)
    # random topological order: repeatedly pick a random ready node
    children = {i: [j for j in range(T) if parent[j] == i] for i in range(-1, T)}
    ready, order = list(children[-1]), []
    while ready:
        x = ready.pop(int(rng.integers(0, len(ready))))
        order.append(x)
        ready.extend(children[x])
    new_of = {old: new for new, old in enumerate(order)}
    parent2 = np.array([-1 if parent[o] < 0 else new_of[parent[o]] for o in order], np.int32)
    perm = np.array(order)
    b2 = make_tree_batch([parent2], b.S_pre, b.q[perm], b.k[perm], b.v[perm], b.gamma[perm],
                         b.beta[perm])
    O2, U2, logP2 = oracle.verify(b2, nthreads=1)
    np.testing.assert_allclose(O2, O[perm], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(U2, U[perm], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(logP2, logP[perm], rtol=1e-14, atol=1e-15)


def test_prefix_causality():
    """Appending nodes never changes the outputs of nodes already in the tree."""
    rng = np.random.default_rng(31)
    parent = I.random_parent_tree(rng, 16, 6)
    b = _random_unit_batch(rng, parent, 5, 4)
    O, U, _ = oracle.verify(b, nthreads=1)
    n = 9
    bs = make_tree_batch([parent[:n]], b.S_pre, b.q[:n], b.k[:n], b.v[:n], b.gamma[:n],
                         b.beta[:n])
    Os, Us, _ = oracle.verify(bs, nthreads=1)
    assert np.array_equal(Os, O[:n]) and np.array_equal(Us, U[:n])


@pytest.mark.parametrize("cfg", [0, 1])
def test_commit_matches_factorised_state(cfg):
    """Eq. (10) evaluated from the oracle's (log P, K, U) reproduces the
    replayed accepted-path state, for every accepted node of the tree."""
    b = I.config_batch(cfg)
    if cfg == 1:  # keep it quick: 4 heads of the single request
        b = make_tree_batch([b.parent], b.S_pre[:, :4], b.q[:, :4], b.k[:, :4], b.v[:, :4],
                            b.gamma[:, :4], b.beta[:, :4])
    O, U, logP = oracle.verify(b)
    for a in list(range(b.N)) + [-1]:
        acc = np.array([a], np.int32)
        S_new = oracle.commit(b, accepted=acc)
        S_fac = commit_from_factors(b, U, logP, accepted=acc)
        assert rel_fro(S_new, S_fac) < 1e-12, a


def test_pack_masks_brute_force():
    rng = np.random.default_rng(41)
    sizes = [1, 7, 33, 64, 65, 128, 0, 5]
    trees = [I.random_parent_tree(rng, T, int(rng.integers(1, 40))) if T else
             np.zeros(0, np.int32) for T in sizes]
    offsets = np.zeros(len(sizes) + 1, np.int32)
    offsets[1:] = np.cumsum(sizes)
    parent = np.concatenate(trees)
    depth, anc, req, st = oracle.pack(offsets, parent, 127)
    assert st == oracle.OK
    for b, par in enumerate(trees):
        sets = ancestors_or_self(par)
        for i, s in enumerate(sets):
            m = anc[offsets[b] + i]
            bits = {32 * w + t for w in range(4) for t in range(32) if (int(m[w]) >> t) & 1}
            assert bits == s
            assert depth[offsets[b] + i] == len(s) - 1
        assert req[b] == (max(len(s) for s in sets) - 1 if sets else 0)


@pytest.mark.parametrize("bad", ["self_parent", "forward_parent", "below_root", "too_big",
                                 "too_deep"])
def test_pack_rejects_bad_topology(bad):
    parent = np.array([-1, 0, 1, 1, 3], np.int32)
    offsets = np.array([0, 5], np.int32)
    max_depth = 8
    expected = oracle.BAD_TOPOLOGY
    if bad == "self_parent":
        parent[3] = 3
    elif bad == "forward_parent":
        parent[2] = 4
    elif bad == "below_root":
        parent[1] = -2
    elif bad == "too_big":
        parent = np.concatenate([[-1], np.arange(0, 129)]).astype(np.int32)
        offsets = np.array([0, 130], np.int32)
    elif bad == "too_deep":
        max_depth = 2
        expected = oracle.DEPTH
    _, _, _, st = oracle.pack(offsets, parent, max_depth)
    assert st == expected


def _slot_layout_path_replay(batch, b, h, a):
    """The accepted node's state written straight in the slot layout [dv][dk]
    (Section IV-D): walking the path root..a, each node applies Eq. (1) to the
    TRANSPOSED state X = S^T,
        X <- gamma X;  u = beta (v - X k);  X <- X + u k^T,
    with X k = S^T k.  Independent of the oracle's [dk][dv] recurrence."""
    o = batch.offsets[b]
    path = []
    j = a
    while j >= 0:
        path.append(j)
        j = int(batch.parent[o + j])
    X = batch.S_pre[b, h].astype(np.float64).T.copy()
    for j in reversed(path):
        kj = batch.k[o + j, h].astype(np.float64)
        vj = batch.v[o + j, h].astype(np.float64)
        X *= float(batch.gamma[o + j, h])
        u = float(batch.beta[o + j, h]) * (vj - X @ kj)
        X += np.outer(u, kj)
    return X


@pytest.mark.parametrize("layout", ["kv", "vk"])
def test_commit_layers_is_each_layers_own_path(layout):
    """Cross-layer commit of three layers sharing one forest: every layer's
    committed slot equals that layer's own path replay (shapes dk=3, dv=5 make
    a transposed layout fail by shape as well as by value); accepted = -1
    leaves the slot at S_pre."""
    base = I.random_batch(seed=41, B=3, H=2, dk=3, dv=5, sizes=[6, 4, 5], max_depth=4,
                          dtype="f32", sigma=0.3, accept="uniform")
    base.accepted[1] = -1
    layers = I.layer_batches(base, 3, seed=9)
    got = oracle.commit_layers(layers, state_layout=layout, nthreads=1)
    assert got.shape == ((3, 3, 2, 3, 5) if layout == "kv" else (3, 3, 2, 5, 3))
    for li, lb in enumerate(layers):
        assert np.array_equal(lb.offsets, base.offsets) and np.array_equal(lb.parent, base.parent)
        for b in range(base.B):
            for h in range(base.H):
                a = int(base.accepted[b])
                exp = (_slot_layout_path_replay(lb, b, h, a) if a >= 0
                       else lb.S_pre[b, h].astype(np.float64).T)
                if layout == "kv":
                    exp = exp.T
                np.testing.assert_allclose(got[li, b, h], exp, rtol=1e-12, atol=1e-13)
    # layers differ (each used its own operands)
    assert not np.allclose(got[0], got[1])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_commit_then_verify_is_the_grafted_tree(seed):
    """The deferred commit's semantics (bole_commit_verify), pinned on the
    oracle: committing the previous round's accepted path and then verifying
    the new tree from the committed state is the same as verifying one tree in
    which the new tree hangs below the accepted node's path -- the path as a
    chain from the old state, the new roots as children of the accepted node.
    The new nodes' outputs agree, their log P differ by log P of the accepted
    node, and committing a new node of either gives the same state."""
    rng = np.random.default_rng(100 + seed)
    H = 2
    prev = I.random_batch(seed=200 + seed, B=1, H=H, dk=4, dv=3, sizes=[9], max_depth=5,
                          dtype="f32", sigma=0.3, accept="deepest")
    cur = I.random_batch(seed=300 + seed, B=1, H=H, dk=4, dv=3, sizes=[7], max_depth=4,
                         dtype="f32", sigma=0.3, accept="uniform")
    # the accepted path, root first
    path, j = [], int(prev.accepted[0])
    while j >= 0:
        path.append(j)
        j = int(prev.parent[j])
    path = path[::-1]
    L, T = len(path), cur.N
    parent = [-1] + list(range(L - 1)) + [(L - 1 if p < 0 else L + p) for p in cur.parent]
    cat = lambda a, b: np.concatenate([a[path], b], axis=0)
    graft = make_tree_batch([parent], prev.S_pre, cat(prev.q, cur.q), cat(prev.k, cur.k),
                            cat(prev.v, cur.v), cat(prev.gamma, cur.gamma),
                            cat(prev.beta, cur.beta))
    O_g, U_g, lp_g = oracle.verify(graft, nthreads=1)
    S1 = oracle.commit(prev, nthreads=1)
    c1 = make_tree_batch([cur.parent], S1, cur.q, cur.k, cur.v, cur.gamma, cur.beta)
    c1.S_pre = S1  # the committed state in fp64, as the grafted tree carries it
    O_c, U_c, lp_c = oracle.verify(c1, nthreads=1)
    np.testing.assert_allclose(O_g[L:], O_c, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(U_g[L:], U_c, rtol=1e-12, atol=1e-14)
    _, _, lp_p = oracle.verify(prev, nthreads=1)
    np.testing.assert_allclose(lp_g[L:], lp_c + lp_p[int(prev.accepted[0])], rtol=1e-12,
                               atol=1e-13)
    x = int(rng.integers(0, T))
    S_g = oracle.commit(graft, accepted=np.array([L + x], np.int32), nthreads=1)
    S_c = oracle.commit(c1, accepted=np.array([x], np.int32), nthreads=1)
    np.testing.assert_allclose(S_g, S_c, rtol=1e-12, atol=1e-14)
