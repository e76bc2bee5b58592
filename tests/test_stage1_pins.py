"""Pins for the stage-1 oracle (tree-parallel short causal convolution, SiLU,
q/k normalisation, gates, convolution-state commit).  Every expected value
comes from a library routine or a closed form, not from the oracle.  CPU only."""
import numpy as np
import pytest

from conftest import make_tree_batch
from gated_deltanet_verification_gb300 import inputs as I
from oracle import stage1


def _batch(parents, H=2, dk=4, dv=3):
    N = sum(len(p) for p in parents)
    z = np.zeros((N, H, dk), np.float32)
    return make_tree_batch(parents, np.zeros((len(parents), H, dk, dv)), z, z,
                           np.zeros((N, H, dv), np.float32), np.ones((N, H)), np.ones((N, H)))


def _inputs(batch, W, seed=3, gate_terms=False):
    return I.stage1_inputs(batch, W=W, seed=seed, dtype="f32", gate_terms=gate_terms)


def _silu(x):
    return x / (1 + np.exp(-x))


def _run(batch, s, **kw):
    return stage1.conv_gates(s.x, s.conv_state, s.conv_w, s.conv_b, s.a, s.b, batch.offsets,
                             batch.parent, batch.H, batch.dk, batch.dv, s.gate_scale,
                             s.gate_bias, **kw)


def _split_norm(y, H, dk, dv):
    N = y.shape[0]
    q = y[:, :H * dk].reshape(N, H, dk)
    k = y[:, H * dk:2 * H * dk].reshape(N, H, dk)
    v = y[:, 2 * H * dk:].reshape(N, H, dv)
    return (q / np.linalg.norm(q, axis=-1, keepdims=True),
            k / np.linalg.norm(k, axis=-1, keepdims=True), v)


@pytest.mark.parametrize("W", [1, 2, 4, 6])
def test_chain_is_token_order_causal_conv(W):
    """A chain tree is an ordinary token sequence after the committed prefix:
    its outputs equal numpy.convolve over [state rows; x rows] per channel."""
    T = 9
    b = _batch([[-1] + list(range(T - 1))])
    s = _inputs(b, W)
    q, k, v, _, _ = _run(b, s)
    seq = np.concatenate([s.conv_state[0].astype(np.float64), s.x.astype(np.float64)])
    C = seq.shape[1]
    y = np.zeros((T, C))
    for c in range(C):
        full = np.convolve(seq[:, c], s.conv_w[c, ::-1].astype(np.float64), mode="full")
        # token t (row W-1+t of seq) reads seq rows t .. t+W-1: full[t + W - 1]
        y[:, c] = full[W - 1:W - 1 + T] + s.conv_b[c]
    qe, ke, ve = _split_norm(_silu(y), b.H, b.dk, b.dv)
    np.testing.assert_allclose(q, qe, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(k, ke, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(v, ve, rtol=1e-12, atol=1e-13)


def test_star_is_one_token_decode_from_the_committed_state():
    """Every child of the committed root sees only the committed prefix:
    y = bias + w[:, W-1] x_i + sum_{d>=1} w[:, W-1-d] state[W-1-d]."""
    W, T = 4, 6
    b = _batch([[-1] * T])
    s = _inputs(b, W)
    q, k, v, _, _ = _run(b, s)
    st = s.conv_state[0].astype(np.float64)
    w = s.conv_w.astype(np.float64)
    y = (s.conv_b + s.x * w[:, W - 1] + (w[:, :W - 1] * st.T).sum(axis=1)).astype(np.float64)
    qe, ke, ve = _split_norm(_silu(y), b.H, b.dk, b.dv)
    np.testing.assert_allclose(v, ve, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(q, qe, rtol=1e-12, atol=1e-13)


def test_sibling_relabelling_permutes_outputs():
    """Renumbering nodes in another parent-before-child order permutes the
    outputs (the window follows parent links, not positions)."""
    par = [-1, 0, 0, 1, 2, 2, 3]
    perm = [0, 2, 1, 5, 4, 3, 6]           # new index -> old index
    inv = np.argsort(perm)
    par2 = [-1 if par[perm[n]] < 0 else int(inv[par[perm[n]]]) for n in range(len(par))]
    assert all(p < n for n, p in enumerate(par2))
    b1 = _batch([par])
    b2 = _batch([par2])
    s1 = _inputs(b1, 4)
    s2 = _inputs(b2, 4)
    s2.x = s1.x[perm]
    s2.a, s2.b = s1.a[perm], s1.b[perm]
    s2.conv_state, s2.conv_w, s2.conv_b = s1.conv_state, s1.conv_w, s1.conv_b
    out1 = _run(b1, s1)
    out2 = _run(b2, s2)
    for x1, x2 in zip(out1, out2):
        np.testing.assert_allclose(x2, x1[perm], rtol=0, atol=0)


def test_gates_closed_form():
    b = _batch([[-1, 0, 1]], H=3)
    s = _inputs(b, 2, gate_terms=True)
    s.a[:] = np.array([0.0, 50.0, -50.0], np.float32)[None, :]
    s.b[:] = np.array([0.0, 40.0, -40.0], np.float32)[None, :]
    s.gate_scale = np.array([1.0, 2.0, 0.5], np.float32)
    s.gate_bias = np.zeros(3, np.float32)
    _, _, _, g, bt = _run(b, s)
    np.testing.assert_allclose(g[:, 0], 0.5, rtol=1e-15)            # exp(-ln 2)
    assert np.all(g[:, 1] < 1e-40)                                  # exp(-2 * 50)
    np.testing.assert_allclose(g[:, 2], np.exp(-0.5 * np.log1p(np.exp(-50.0))), rtol=1e-15)
    np.testing.assert_allclose(bt[:, 0], 0.5, rtol=1e-15)
    np.testing.assert_allclose(bt[:, 1], 1.0, rtol=1e-15)
    assert np.all(bt[:, 2] < 1e-17)
    # gate bias shifts the pre-activation: a + c = 0 gives exp(-s ln 2)
    s.a[:] = 1.5
    s.gate_bias = np.full(3, -1.5, np.float32)
    _, _, _, g, _ = _run(b, s)
    exp = np.exp(-s.gate_scale.astype(np.float64) * np.log(2.0))
    np.testing.assert_allclose(g, np.broadcast_to(exp, g.shape), rtol=1e-14)


@pytest.mark.parametrize("W", [2, 4, 5])
def test_conv_commit_matches_token_order_window(W):
    """Committing node a of a chain keeps the last W-1 rows of
    [old state; x_0 .. x_a]; a = -1 keeps the state."""
    T = 6
    b = _batch([[-1] + list(range(T - 1))] * 3)
    s = _inputs(b, W)
    acc = np.array([0, T - 1, -1], np.int32)
    new = stage1.conv_commit(s.conv_state, s.x, b.offsets, b.parent, acc)
    for r, a in enumerate(acc):
        if a < 0:
            assert np.array_equal(new[r], s.conv_state[r])
            continue
        o = b.offsets[r]
        seq = np.concatenate([s.conv_state[r], s.x[o:o + a + 1]])
        assert np.array_equal(new[r], seq[-(W - 1):])


def test_conv_commit_on_a_branch_skips_siblings():
    """The committed window follows the accepted node's ancestors only."""
    par = [-1, 0, 0, 2, 1]                 # node 3's path: 0 -> 2 -> 3
    b = _batch([par])
    s = _inputs(b, 4)
    new = stage1.conv_commit(s.conv_state, s.x, b.offsets, b.parent, np.array([3], np.int32))
    assert np.array_equal(new[0], s.x[[0, 2, 3]])
    new = stage1.conv_commit(s.conv_state, s.x, b.offsets, b.parent, np.array([2], np.int32))
    assert np.array_equal(new[0], np.stack([s.conv_state[0][2], s.x[0], s.x[2]]))


# ---- planted mistakes: each must fail at least one pin above ----
STAGE1_MUTANTS = {
    "weight_not_flipped": ("acc += w[:, W - 1 - dist] * row", "acc += w[:, dist] * row"),
    "previous_index_not_parent": ("j = int(parent_local[j])", "j = j - 1"),
    "no_silu": ("y[o + i] = _silu(acc)", "y[o + i] = acc"),
    "state_rows_reversed": ("row = x[o + tok] if tok >= 0 else st[r, -tok - 1]",
                            "row = x[o + tok] if tok >= 0 else st[r, W - 2 - (-tok - 1)]"),
    "no_bias": ("acc = bias.copy()", "acc = np.zeros(C)"),
    "gate_bias_outside": ("_softplus(a + gbias[None, :])", "(_softplus(a) + gbias[None, :])"),
    "commit_oldest_first": ("st[r, Wm1 - 1 - pos] =", "st[r, pos] ="),
}


def _stage1_pins_pass(mod) -> bool:
    saved = stage1.__dict__.copy()
    try:
        stage1.conv_gates, stage1.conv_commit = mod.conv_gates, mod.conv_commit
        tests = [lambda: test_chain_is_token_order_causal_conv(4),
                 test_star_is_one_token_decode_from_the_committed_state,
                 test_sibling_relabelling_permutes_outputs, test_gates_closed_form,
                 lambda: test_conv_commit_matches_token_order_window(4),
                 test_conv_commit_on_a_branch_skips_siblings]
        for t in tests:
            try:
                t()
            except AssertionError:
                return False
        return True
    finally:
        stage1.conv_gates, stage1.conv_commit = saved["conv_gates"], saved["conv_commit"]


def test_unmodified_stage1_oracle_passes():
    assert _stage1_pins_pass(stage1)


@pytest.mark.parametrize("name", sorted(STAGE1_MUTANTS))
def test_stage1_mutant_is_caught(name):
    import types
    old, new = STAGE1_MUTANTS[name]
    src = open(stage1.__file__).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType(f"stage1_{name}")
    exec(compile(src.replace(old, new), f"stage1_{name}", "exec"), mod.__dict__)
    assert not _stage1_pins_pass(mod), f"pins did not catch {name}"
