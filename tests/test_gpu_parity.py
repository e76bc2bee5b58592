"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle,
on the same seeded inputs.  Integer outputs must match bit for bit; O, U and
the committed state within relative Frobenius 1e-5 (float32 q/k/v) or 1e-2
(bf16 q/k/v, float32 state).  logP is compared with an absolute bound
derived from float32 summation of at most 128 logs (|L| < 200 here)."""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_local_parity, rel_fro, state_unit_errors
from gated_deltanet_verification_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_verification_gb300 import build
    build.build()


def _run(batch, flags=0, dtype=None):
    from gated_deltanet_verification_gb300 import bole, device
    db = device.to_device(batch, dtype=dtype)
    rb = device.alloc_round(db, flags)
    device.pack(db, rb)
    device.verify(db, rb, flags)
    O = rb.O.float().cpu().numpy().astype(np.float64)
    U = rb.U.cpu().numpy().astype(np.float64)
    logP = rb.logP.cpu().numpy().astype(np.float64)
    device.commit(db, rb, flags)
    S_new = db.S.cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    bole.check_status(rb.status)
    return dict(depth=rb.depth.cpu().numpy(), anc=rb.anc.cpu().numpy().view(np.uint32),
                req=rb.req_depth[:batch.B].cpu().numpy(), O=O, U=U, logP=logP, S_new=S_new)


def _check(batch, got, tol):
    """Integers bit for bit; O, U and S_new within `tol` as whole tensors, per
    (request, head) and per node row (Theorem 1 is an equality per node, so a
    wrong node or head must not hide inside a large tensor's norm)."""
    depth, anc, req, st = oracle.pack(batch.offsets, batch.parent, batch.max_depth)
    assert st == oracle.OK
    assert np.array_equal(got["depth"], depth)
    assert np.array_equal(got["anc"], anc)
    assert np.array_equal(got["req"], req)
    O, U, logP = oracle.verify(batch)
    S_new = oracle.commit(batch)
    errs = {"O": rel_fro(got["O"], O), "U": rel_fro(got["U"], U),
            "S_new": rel_fro(got["S_new"], S_new)}
    assert np.max(np.abs(got["logP"] - logP)) < 2e-4 * max(1.0, np.max(np.abs(logP)))
    for name, e in errs.items():
        assert e <= tol, f"{batch.name}: {name} rel err {e:.3e} > {tol}"
    for name, ref in (("O", O), ("U", U)):
        unit, row = assert_local_parity(batch.name, name, got[name], ref, batch.offsets, tol)
        errs[name + "_worst_head"], errs[name + "_worst_row"] = unit, row
    su = state_unit_errors(got["S_new"], S_new)
    (wb, wh), worst = max(su.items(), key=lambda kv: kv[1])
    assert worst <= tol, f"{batch.name}: S_new worst (request, head) = ({wb}, {wh}) {worst:.3e}"
    errs["S_new_worst_head"] = worst
    return errs


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_config_parity(cfg):
    b = I.config_batch(cfg)
    errs = _check(b, _run(b), TOL[b.dtype])
    print(b.name, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("shape", I.SHAPES_CFG4)
def test_shape_extremes_parity(shape):
    b = I.config_batch(4, shape=shape)
    errs = _check(b, _run(b), TOL[b.dtype])
    print(b.name, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("cfg", [1, 2])
def test_cuda_core_path_parity(cfg):
    """The FP32 CUDA-core kernels on the bf16 workloads (forced)."""
    from gated_deltanet_verification_gb300 import bole
    b = I.config_batch(cfg)
    _check(b, _run(b, flags=bole.FLAG_FORCE_SIMT), TOL["bf16"])


@pytest.mark.parametrize("cfg", [1, 2])
def test_fp32_inputs_parity(cfg):
    """Same workloads with full-precision float32 q/k/v (the tensor-core
    value-tiled kernel, three-way bf16 operand split): float32 tolerance."""
    b = I.config_batch(cfg, dtype="f32")
    errs = _check(b, _run(b, dtype=torch.float32), TOL["f32"])
    print(b.name, "f32", {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("sizes,H,max_depth,shape,sigma", [
    ([32] * 8, 8, 8, "random", 0.05),         # the batched forest's shape
    ([1, 32, 0, 7, 0, 2], 3, 15, "random", 0.1),  # 1-node, empty and ragged trees
    ([16, 16, 9], 5, 15, "chain", 0.1),        # the deepest chains the kernel takes
    ([32, 32], 2, 1, "star", 0.1),             # depth 0
    ([24, 31], 4, 15, "random", 0.5),          # large operands: the split's lower copies carry weight
])
def test_fp32_tensor_core_kernel_matches_oracle_and_cuda_core(sizes, H, max_depth, shape, sigma):
    """fp32 q/k/v on the tensor cores: every fp32 operand of the Gram and the
    state products as three bf16 parts (six products kept), the propagation
    as tf32 hi + lo.  Against the oracle per tensor, per (request, head) and
    per node row at the float32 bound, and against the FP32 CUDA-core kernels
    (FLAG_FORCE_SIMT) on the same forest."""
    from gated_deltanet_verification_gb300 import bole
    b = I.random_batch(seed=sum(sizes) + 11 * H, B=len(sizes), H=H, dk=128, dv=128, sizes=sizes,
                       max_depth=max_depth, dtype="f32", sigma=sigma, shape=shape,
                       accept="uniform")
    Oe, Ue, Le = oracle.verify(b)
    Se = oracle.commit(b)
    got = {}
    for name, flags in (("tc", 0), ("simt", bole.FLAG_FORCE_SIMT)):
        O, U, logP, S_new = _verify_flags(b, flags, max_T=32, commit=True)
        assert rel_fro(O, Oe) <= TOL["f32"] and rel_fro(U, Ue) <= TOL["f32"], name
        assert_local_parity(f"{b.name}/{name}", "O", O, Oe, b.offsets, TOL["f32"])
        assert_local_parity(f"{b.name}/{name}", "U", U, Ue, b.offsets, TOL["f32"])
        assert np.max(np.abs(logP - Le)) < 2e-4 * max(1.0, np.max(np.abs(Le)))
        # commit (fp32 keys: tf32 hi + lo operands on the tensor-core path)
        assert max(state_unit_errors(S_new, Se).values()) <= TOL["f32"], name
        got[name] = (O, U, S_new)
    for t in range(3):
        assert rel_fro(got["tc"][t], got["simt"][t]) <= 1e-5


@pytest.mark.parametrize("sizes,shape,dtype,dk,dv,max_depth", [
    ([1, 2, 63, 64, 65, 128], "random", "f32", 32, 48, 9),
    ([1, 2, 63, 64], "random", "bf16", 128, 128, 9),
    ([64, 0, 17, 0, 64], "chain", "bf16", 128, 128, 127),
    ([32, 20, 5, 1], "chain", "bf16", 128, 128, 31),
    ([16, 9, 12], "chain", "bf16", 128, 128, 15),
    ([64, 7], "star", "bf16", 128, 128, 1),
    ([64, 50, 21], "4ary", "bf16", 128, 128, 3),
    ([5, 0, 3], "star", "f32", 16, 16, 1),
    ([128, 100], "4ary", "bf16", 64, 128, 3),
    ([40, 33, 64], "random", "bf16", 128, 128, 12),
    ([64] * 20, "random", "bf16", 128, 128, 30),
    ([64] * 20, "random", "bf16", 128, 128, 15),
    ([1, 32, 1, 7], "random", "bf16", 128, 128, 15),   # small-tree layout, 1-node trees
    ([128, 1, 2], "chain", "bf16", 128, 128, 127),    # large-tree kernel, depths 127 and 0
])
def test_ragged_and_edge_shapes(sizes, shape, dtype, dk, dv, max_depth):
    b = I.random_batch(seed=sum(sizes) + dk, B=len(sizes), H=3, dk=dk, dv=dv, sizes=sizes,
                       max_depth=max_depth, dtype=dtype, sigma=0.05, accept="uniform",
                       shape=shape)
    _check(b, _run(b), TOL[dtype])


@pytest.mark.parametrize("which", ["none", "root_child"])
def test_commit_edge_paths(which):
    b = I.random_batch(seed=3, B=3, H=2, dk=128, dv=128, sizes=[20, 31, 9], max_depth=6,
                       dtype="bf16", sigma=0.05, accept="uniform")
    b.accepted[:] = -1 if which == "none" else 0
    got = _run(b)
    S_new = oracle.commit(b)
    assert rel_fro(got["S_new"], S_new) <= TOL["bf16"]
    assert max(state_unit_errors(got["S_new"], S_new).values()) <= TOL["bf16"]
    if which == "none":
        assert np.array_equal(got["S_new"], b.S_pre.astype(np.float64))


def _node_depths(parent):
    """Depth of every node of one parent-before-child tree (root depth 0)."""
    d = []
    for p in parent:
        d.append(0 if p < 0 else d[p] + 1)
    return d


@pytest.mark.parametrize("shape", ["chain", "spine"])
def test_commit_long_accepted_paths(shape):
    """Accepted paths of more than one 16-node product chunk: 17, 33, 64 and
    128 nodes in trees of more than 32 nodes (the walker's first chunk, then
    pointer jumping over the ancestor masks; the rows staged two chunks
    ahead) and 20 nodes in a 30-node tree (walked serially, rows staged); on
    spines with side branches the deepest node of each."""
    if shape == "chain":
        b = I.random_batch(seed=71, B=5, H=2, dk=128, dv=128, sizes=[128, 40, 64, 100, 30],
                           max_depth=127, dtype="bf16", sigma=0.05, shape="chain")
        b.accepted[:] = [127, 16, 32, 63, 19]
    else:  # a spine with side branches: path nodes are not consecutive indices
        rng = np.random.default_rng(72)
        trees = []
        for T in (128, 96, 70, 128):
            par, tip = [-1], 0
            for i in range(1, T):
                if rng.random() < 0.6:
                    par.append(tip)
                    tip = i
                else:
                    par.append(int(rng.integers(0, i)))
            trees.append(np.asarray(par, np.int32))
        depth = max(max(_node_depths(t)) for t in trees)
        b = I.make_batch("spine72", rng, trees, 2, 128, 128, "bf16", depth, 0.05, "deepest")
        assert min(_node_depths(t)[b.accepted[i]] for i, t in enumerate(trees)) >= 16
    _check(b, _run(b), TOL["bf16"])


@pytest.mark.parametrize("bad_parent", [45, -7])
def test_commit_reports_a_bad_link_deep_on_the_path(bad_parent):
    """A parent link that is not backwards 24 nodes up a 64-node accepted
    path (found by pointer jumping, not by the walker's first chunk): the
    commit reports {BOLE_ERR_BAD_TOPOLOGY, request, node, -1} and leaves that
    request's state as it was; the other request is committed."""
    from gated_deltanet_verification_gb300 import bole, device
    b = I.random_batch(seed=73, B=2, H=2, dk=128, dv=128, sizes=[64, 40], max_depth=63,
                       dtype="bf16", sigma=0.05, shape="chain")
    b.accepted[:] = [63, 30]
    db = device.to_device(b)
    rb = device.alloc_round(db)
    device.pack(db, rb)
    device.verify(db, rb, 0)
    torch.cuda.synchronize()
    bole.check_status(rb.status)
    S0 = db.S.clone()
    bad = torch.as_tensor(b.parent.copy(), device="cuda")
    bad[40] = bad_parent  # node 40 of request 0
    st = bole.new_status()
    bole.commit(db.S, db.k, rb.U, rb.logP, db.offsets, bad, db.accepted, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [bole.ERR_BAD_TOPOLOGY, 0, 40, -1]
    assert torch.equal(db.S[0], S0[0])
    S_new = oracle.commit(b)
    su = state_unit_errors(db.S.cpu().numpy().astype(np.float64), S_new)
    assert max(su[(1, h)] for h in range(b.H)) <= TOL["bf16"]


def test_device_topology_faults():
    """Bad parents and over-deep trees are reported in the status block; the
    verification and commit kernels then leave their outputs untouched."""
    from gated_deltanet_verification_gb300 import bole, device
    b = I.random_batch(seed=5, B=2, H=2, dk=128, dv=128, sizes=[12, 9], max_depth=4,
                       dtype="bf16", sigma=0.05, accept="uniform")
    bad = b.parent.copy()
    bad[12 + 4] = 7  # node 4 of request 1 points forward
    db = device.to_device(b)
    db.parent.copy_(torch.from_numpy(bad))
    rb = device.alloc_round(db)
    rb.O.fill_(3.0)
    S_before = db.S.clone()
    device.run_round(db, rb)
    torch.cuda.synchronize()
    st = rb.status.cpu().tolist()
    assert st[0] == bole.ERR_BAD_TOPOLOGY and st[1] == 1 and st[2] == 4
    assert torch.all(rb.O.float() == 3.0)
    assert torch.equal(db.S, S_before)
    # depth bound violated
    db2 = device.to_device(b)
    db2.max_depth = 1
    rb2 = device.alloc_round(db2)
    device.pack(db2, rb2)
    torch.cuda.synchronize()
    st2 = rb2.status.cpu().tolist()
    assert st2[0] == bole.ERR_DEPTH
    with pytest.raises(bole.BoleError):
        bole.check_status(rb2.status)


def test_empty_batch():
    from gated_deltanet_verification_gb300 import bole
    offsets = torch.zeros(1, dtype=torch.int32, device="cuda")
    parent = torch.zeros(0, dtype=torch.int32, device="cuda")
    depth, anc, req, st = bole.pack_forest(offsets, parent, 3)
    torch.cuda.synchronize()
    assert st.cpu().tolist()[0] == 0


def test_overlapped_round_matches_serial_launches():
    """run_round overlaps verify with pack and commit with verify (programmatic
    dependent launch); the results must equal those of fully serial launches
    bit for bit, and match the oracle."""
    from gated_deltanet_verification_gb300 import bole, device
    for cfg in (2, 3):
        b = I.config_batch(cfg)
        db1, db2 = device.to_device(b), device.to_device(b)
        rb1, rb2 = device.alloc_round(db1), device.alloc_round(db2)
        device.pack(db1, rb1)
        device.verify(db1, rb1)
        device.commit(db1, rb1)
        device.run_round(db2, rb2)
        torch.cuda.synchronize()
        bole.check_status(rb1.status)
        bole.check_status(rb2.status)
        assert torch.equal(rb1.O, rb2.O)
        assert torch.equal(rb1.U, rb2.U)
        assert torch.equal(rb1.logP, rb2.logP)
        assert torch.equal(db1.S, db2.S)
    got = dict(depth=rb2.depth.cpu().numpy(), anc=rb2.anc.cpu().numpy().view(np.uint32),
               req=rb2.req_depth[:b.B].cpu().numpy(),
               O=rb2.O.float().cpu().numpy().astype(np.float64),
               U=rb2.U.cpu().numpy().astype(np.float64),
               logP=rb2.logP.cpu().numpy().astype(np.float64),
               S_new=db2.S.cpu().numpy().astype(np.float64))
    _check(b, got, 1e-2)


@pytest.mark.parametrize("seed,sizes,depth", [(31, [100, 70], 40), (32, [128], 127), (33, [48], 20),
                                              (34, [80, 128], 0)])
def test_large_tree_factors_match_dense_inverse(seed, sizes, depth):
    """The large-tree kernel keeps [M; W] = [C (I+G)^{-1}; (I+G)^{-1}] in tensor
    memory and needs no workspace; given one of B H 256 128 floats it also
    writes [M; W] there (depth 0, the stars: M = diag(q_i . k_i), W = I,
    formed on the CUDA cores).  Compare with a library dense inverse of the same G
    and C (Lemma 3: the log-depth product of (I + G^(2^k)) equals the finite
    Neumann sum), and O, U with the oracle."""
    from gated_deltanet_verification_gb300 import bole, device
    import pins_lib
    shape = "chain" if depth >= 100 else "star" if depth == 0 else "random"
    b = I.random_batch(seed=seed, B=len(sizes), H=2, dk=128, dv=128, sizes=sizes,
                       max_depth=max(depth, 1), dtype="bf16", sigma=0.05, shape=shape)
    db = device.to_device(b)
    rb = device.alloc_round(db)
    assert bole.workspace_size(b.B, b.H, 128, 128, b.max_T, b.max_depth, db.q.dtype, 0) == 0
    rb.workspace = torch.full((b.B * b.H * 256 * 128,), float("nan"), dtype=torch.float32,
                              device="cuda")
    device.pack(db, rb)
    device.verify(db, rb)
    torch.cuda.synchronize()
    bole.check_status(rb.status)
    Oe, Ue, _ = oracle.verify(b)
    assert rel_fro(rb.O.float().cpu().numpy(), Oe) <= TOL["bf16"]
    assert rel_fro(rb.U.cpu().numpy(), Ue) <= TOL["bf16"]
    assert_local_parity(b.name, "O", rb.O.float().cpu().numpy(), Oe, b.offsets, TOL["bf16"])
    assert_local_parity(b.name, "U", rb.U.cpu().numpy(), Ue, b.offsets, TOL["bf16"])
    mw = rb.workspace.view(b.B, b.H, 256, 128).cpu().numpy()
    for r in range(b.B):
        o, e = int(b.offsets[r]), int(b.offsets[r + 1])
        T = e - o
        for hh in range(b.H):
            # G, C with decay ratios taken in log space (a 128-node chain underflows P)
            anc = pins_lib.ancestors_or_self(b.parent[o:e])
            lg = np.log(b.gamma[o:e, hh].astype(np.float64))
            L = np.array([sum(lg[j] for j in anc[i]) for i in range(T)])
            q64 = b.q[o:e, hh].astype(np.float64)
            k64 = b.k[o:e, hh].astype(np.float64)
            G = np.zeros((T, T))
            C = np.zeros((T, T))
            for i in range(T):
                for j in anc[i]:
                    ratio = np.exp(L[i] - L[j])
                    C[i, j] = ratio * (q64[i] @ k64[j])
                    if j != i:
                        G[i, j] = b.beta[o + i, hh] * ratio * (k64[i] @ k64[j])
            W = np.linalg.inv(np.eye(T) + G)
            M = C @ W
            Wg = mw[r, hh, 128:128 + T, :T]
            Mg = mw[r, hh, :T, :T]
            assert rel_fro(Wg, W) < 5e-3, (r, hh, rel_fro(Wg, W))
            assert rel_fro(Mg, M) < 5e-3, (r, hh, rel_fro(Mg, M))
            # padding rows and columns stay exactly zero (W keeps its unit diagonal)
            assert np.all(mw[r, hh, :T, T:] == 0) and np.all(mw[r, hh, 128:128 + T, T:] == 0)


def _verify_direct(b, max_T):
    from gated_deltanet_verification_gb300 import bole
    def t(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dt)
    offsets, parent = t(b.offsets, torch.int32), t(b.parent, torch.int32)
    depth, anc, req, st = bole.pack_forest(offsets, parent, b.max_depth)
    O, U, logP = bole.tree_verify(t(b.S_pre, torch.float32), t(b.q, torch.bfloat16),
                                  t(b.k, torch.bfloat16), t(b.v, torch.bfloat16),
                                  t(b.gamma, torch.float32), t(b.beta, torch.float32), offsets,
                                  parent, depth, anc, req, max_T, b.max_depth, status=st)
    torch.cuda.synchronize()
    return (O.float().cpu().numpy().astype(np.float64), U.cpu().numpy().astype(np.float64),
            logP.cpu().numpy().astype(np.float64), st.cpu().tolist())


def test_small_tree_layout_matches_the_64_node_layout():
    """A forest whose trees hold at most 32 nodes runs the small-tree layout of
    the fused kernel (value rows and Gram in the [Q;K] padding, factors formed
    beside the state products); declaring max_T = 64 runs the 64-node layout
    on the same forest.  Both against the oracle, and against each other
    (same products, same substitution order)."""
    b = I.random_batch(seed=91, B=7, H=3, dk=128, dv=128, sizes=[32, 1, 17, 0, 32, 9, 25],
                       max_depth=15, dtype="bf16", sigma=0.05, shape="random")
    Oe, Ue, _ = oracle.verify(b)
    got = []
    for max_T in (32, 64):
        O, U, logP, st = _verify_direct(b, max_T)
        assert st[0] == 0, st
        assert rel_fro(O, Oe) <= TOL["bf16"] and rel_fro(U, Ue) <= TOL["bf16"]
        assert_local_parity(b.name, "O", O, Oe, b.offsets, TOL["bf16"])
        assert_local_parity(b.name, "U", U, Ue, b.offsets, TOL["bf16"])
        got.append((O, U, logP))
    assert rel_fro(got[0][1], got[1][1]) <= 1e-5
    assert rel_fro(got[0][0], got[1][0]) <= 1e-4  # bf16 rounding of equal fp32 values
    assert np.array_equal(got[0][2], got[1][2])


def test_tree_above_declared_max_T_is_reported():
    """max_T bounds every tree: a 33-node tree declared as max_T = 32 is
    reported as a topology error by the small-tree kernel, which then loads
    none of its operands and writes no output."""
    from gated_deltanet_verification_gb300 import bole
    b = I.random_batch(seed=92, B=2, H=2, dk=128, dv=128, sizes=[5, 33], max_depth=6,
                       dtype="bf16", sigma=0.05)
    _, _, _, st = _verify_direct(b, 32)
    assert st[0] == bole.ERR_BAD_TOPOLOGY and st[1] == 1, st


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """Failure detection without a fault: a device thread waits on a barrier
    nothing arrives on; the bounded wait gives up after the limit, reports
    BOLE_ERR_TIMEOUT with the time waited, and the next calls on the same
    context run normally (a verification and commit against the oracle)."""
    from gated_deltanet_verification_gb300 import bole
    for limit_ms in (2, 20):
        st = bole.selftest_wait(limit_ms * 1_000_000)
        torch.cuda.synchronize()
        code, req, node, waited_us = st.cpu().tolist()
        assert (code, req, node) == (bole.ERR_TIMEOUT, -1, -1)
        assert limit_ms * 1000 <= waited_us < limit_ms * 1000 + 50_000
        with pytest.raises(bole.BoleError):
            bole.check_status(st)
    b = I.random_batch(seed=97, B=3, H=2, dk=128, dv=128, sizes=[20, 31, 9], max_depth=6,
                       dtype="bf16", sigma=0.05, accept="uniform")
    _check(b, _run(b), TOL["bf16"])


def _verify_flags(b, flags, max_T=None, commit=False):
    from gated_deltanet_verification_gb300 import bole, device
    db = device.to_device(b)
    if max_T is not None:
        db.max_T = max_T
    rb = device.alloc_round(db, flags)
    device.pack(db, rb)
    device.verify(db, rb, flags)
    if commit:
        device.commit(db, rb, flags)
    torch.cuda.synchronize()
    bole.check_status(rb.status)
    out = (rb.O.float().cpu().numpy().astype(np.float64), rb.U.cpu().numpy().astype(np.float64),
           rb.logP.cpu().numpy().astype(np.float64))
    return out + (db.S.cpu().numpy().astype(np.float64),) if commit else out


@pytest.mark.parametrize("sizes,H,max_depth,shape", [
    ([32] * 16, 32, 8, "random"),          # the batched forest's shape
    ([1, 32, 0, 7, 0, 2], 3, 15, "random"),  # 1-node, empty and ragged trees, odd head count
    ([16, 16, 9], 5, 15, "chain"),         # the deepest chains the kernel takes (depth 15)
    ([32, 32], 2, 1, "star"),              # depth 0: no propagation
])
def test_value_tiled_kernel_matches_oracle_and_one_tile_per_head(sizes, H, max_depth, shape):
    """Trees of up to 32 nodes: BOLE_FLAG_VALUE_TILES runs the value-tiled
    kernel (two CTAs per head, 64 value columns each, Section IV-B),
    BOLE_FLAG_ONE_TILE_PER_HEAD the one-CTA-per-head kernel on the same forest.  Both against the oracle per
    tensor, per (request, head) and per node row, and against each other (the
    same products; only the propagation's accumulation differs)."""
    from gated_deltanet_verification_gb300 import bole
    b = I.random_batch(seed=sum(sizes) + 7 * H, B=len(sizes), H=H, dk=128, dv=128, sizes=sizes,
                       max_depth=max_depth, dtype="bf16", sigma=0.05, shape=shape)
    Oe, Ue, Le = oracle.verify(b)
    got = {}
    for name, flags in (("vtile", bole.FLAG_VALUE_TILES), ("one_tile", bole.FLAG_ONE_TILE_PER_HEAD)):
        O, U, logP = _verify_flags(b, flags, max_T=32)
        assert rel_fro(O, Oe) <= TOL["bf16"] and rel_fro(U, Ue) <= TOL["bf16"], name
        assert_local_parity(f"{b.name}/{name}", "O", O, Oe, b.offsets, TOL["bf16"])
        assert_local_parity(f"{b.name}/{name}", "U", U, Ue, b.offsets, TOL["bf16"])
        assert np.max(np.abs(logP - Le)) < 2e-4 * max(1.0, np.max(np.abs(Le)))
        got[name] = (O, U, logP)
    assert rel_fro(got["vtile"][1], got["one_tile"][1]) <= 1e-5
    assert rel_fro(got["vtile"][0], got["one_tile"][0]) <= 1e-4
    assert np.array_equal(got["vtile"][2], got["one_tile"][2])


@pytest.mark.parametrize("cfg", [1, 2])
def test_value_tiled_round_matches_serial_and_one_tile_commit(cfg):
    """A whole overlapped round (pack -> value-tiled verify -> commit with
    programmatic dependent launch) equals serial launches bit for bit and
    commits the oracle's state (config 1 takes the value tiles by default)."""
    from gated_deltanet_verification_gb300 import bole, device
    b = I.config_batch(cfg)
    f = bole.FLAG_VALUE_TILES
    db1, db2 = device.to_device(b), device.to_device(b)
    rb1, rb2 = device.alloc_round(db1), device.alloc_round(db2)
    device.pack(db1, rb1)
    device.verify(db1, rb1, f)
    device.commit(db1, rb1)
    device.run_round(db2, rb2, f)
    torch.cuda.synchronize()
    bole.check_status(rb1.status)
    bole.check_status(rb2.status)
    assert torch.equal(rb1.O, rb2.O) and torch.equal(rb1.U, rb2.U)
    assert torch.equal(db1.S, db2.S)
    S_new = oracle.commit(b)
    assert max(state_unit_errors(db2.S.cpu().numpy(), S_new).values()) <= TOL["bf16"]


@pytest.mark.parametrize("cfg,extra", [(1, 0), (2, 0), (3, 0), (2, "vt"), (3, "vk"), (2, "f32")])
def test_inline_topology_round_matches_pack_round(cfg, extra):
    """BOLE_FLAG_INLINE_TOPOLOGY: the verification forms each node's ancestor
    mask and depth from the parent links itself (no bole_pack_forest); the
    round's O, U, log P and committed state are bit-identical to the round
    with pack, on both small-tree kernels (bf16 and fp32 q/k/v) and the
    [dv, dk] slot layout."""
    from gated_deltanet_verification_gb300 import bole, device
    b = I.config_batch(cfg, dtype="f32" if extra == "f32" else None)
    f = bole.FLAG_VALUE_TILES if extra == "vt" else 0
    db1, db2 = device.to_device(b), device.to_device(b)
    if extra == "vk":
        f = bole.FLAG_STATE_VK
        for db in (db1, db2):
            db.S = db.S.transpose(2, 3).contiguous()
    rb1, rb2 = device.alloc_round(db1, f), device.alloc_round(db2, f)
    device.run_round(db1, rb1, f)
    device.pack(db2, rb2)  # the topology outputs are not used below: zero them
    rb2.depth.zero_(); rb2.anc.zero_(); rb2.req_depth.zero_(); rb2.status.zero_()
    bole.tree_verify(db2.S, db2.q, db2.k, db2.v, db2.gamma, db2.beta, db2.offsets, db2.parent,
                     None, None, None, db2.max_T, db2.max_depth, O=rb2.O, U=rb2.U,
                     logP=rb2.logP, status=rb2.status,
                     flags=f | bole.FLAG_INLINE_TOPOLOGY | bole.FLAG_OVERLAP_LAUNCH)
    device.commit(db2, rb2, f | bole.FLAG_OVERLAP_LAUNCH)
    torch.cuda.synchronize()
    bole.check_status(rb1.status)
    bole.check_status(rb2.status)
    assert torch.equal(rb1.O, rb2.O) and torch.equal(rb1.U, rb2.U)
    assert torch.equal(rb1.logP, rb2.logP) and torch.equal(db1.S, db2.S)
    if cfg == 3 and not extra:
        got = dict(depth=rb1.depth.cpu().numpy(), anc=rb1.anc.cpu().numpy().view(np.uint32),
                   req=rb1.req_depth[:b.B].cpu().numpy(),
                   O=rb2.O.float().cpu().numpy().astype(np.float64),
                   U=rb2.U.cpu().numpy().astype(np.float64),
                   logP=rb2.logP.cpu().numpy().astype(np.float64),
                   S_new=db2.S.cpu().numpy().astype(np.float64))
        _check(b, got, TOL["bf16"])


@pytest.mark.parametrize("vt", [False, True, "f32"])
def test_inline_topology_faults_and_sticky_status(vt):
    """Faults found by the in-kernel topology step: a forward link is reported
    with its request, node and parent and that request's outputs stay
    unwritten (the commit then writes nothing); a tree deeper than max_depth
    is reported as a depth error; the status block is not cleared by the next
    round, which writes nothing until the caller zeroes it.  On the one-CTA
    kernel, the value tiles and the fp32 value tiles."""
    from gated_deltanet_verification_gb300 import bole, device
    f = bole.FLAG_INLINE_TOPOLOGY | (bole.FLAG_VALUE_TILES if vt is True else 0)
    dtype = "f32" if vt == "f32" else "bf16"
    b = I.random_batch(seed=55, B=3, H=2, dk=128, dv=128, sizes=[12, 9, 20], max_depth=6,
                       dtype=dtype, sigma=0.05, accept="uniform")
    bad = b.parent.copy()
    bad[12 + 5] = 8  # node 5 of request 1 points forward
    db = device.to_device(b)
    db.parent.copy_(torch.from_numpy(bad))
    rb = device.alloc_round(db, f)
    rb.O.fill_(3.0)
    S0 = db.S.clone()
    device.run_round(db, rb, f)
    torch.cuda.synchronize()
    assert rb.status.cpu().tolist() == [bole.ERR_BAD_TOPOLOGY, 1, 5, 8]
    assert torch.all(rb.O[12:21].float() == 3.0)          # the bad request: untouched
    assert not torch.all(rb.O[0:12].float() == 3.0)       # the others verified
    assert torch.equal(db.S, S0)                          # the commit wrote nothing
    # sticky: a clean forest verifies nothing until the status is zeroed
    db.parent.copy_(torch.from_numpy(b.parent))
    rb.O.fill_(3.0)
    device.run_round(db, rb, f)
    torch.cuda.synchronize()
    assert rb.status.cpu().tolist()[0] == bole.ERR_BAD_TOPOLOGY
    assert torch.all(rb.O.float() == 3.0) and torch.equal(db.S, S0)
    rb.status.zero_()
    device.run_round(db, rb, f)
    torch.cuda.synchronize()
    bole.check_status(rb.status)
    S_new = oracle.commit(b)
    assert max(state_unit_errors(db.S.cpu().numpy(), S_new).values()) <= TOL[dtype]
    # depth above the declared bound
    db2 = device.to_device(b)
    db2.max_depth = 2
    rb2 = device.alloc_round(db2, f)
    device.run_round(db2, rb2, f)
    torch.cuda.synchronize()
    st = rb2.status.cpu().tolist()
    assert st[0] == bole.ERR_DEPTH and st[2] == -1 and st[3] > 2


def test_inline_topology_unsupported_paths():
    """Kernels that read the masks bole_pack_forest builds (the large-tree
    kernel, the CUDA-core kernels) refuse the flag synchronously."""
    from gated_deltanet_verification_gb300 import bole, device
    b = I.random_batch(seed=56, B=2, H=2, dk=128, dv=128, sizes=[40, 70], max_depth=30,
                       dtype="bf16", sigma=0.05)
    db = device.to_device(b)
    rb = device.alloc_round(db)
    for flags in (bole.FLAG_INLINE_TOPOLOGY,
                  bole.FLAG_INLINE_TOPOLOGY | bole.FLAG_FORCE_SIMT):
        with pytest.raises(bole.BoleError) as e:
            bole.tree_verify(db.S, db.q, db.k, db.v, db.gamma, db.beta, db.offsets, db.parent,
                             None, None, None, db.max_T, db.max_depth, status=rb.status,
                             workspace=rb.workspace, flags=flags)
        assert e.value.code == bole.ERR_UNSUPPORTED
