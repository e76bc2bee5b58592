"""A seeded sweep over random forests: request counts, head counts, tree
sizes from empty to 128 nodes, tree shapes, q/k/v dtypes and the flags that
choose between the verification kernels (default choice, value tiles, one CTA
per head, the topology step inside the verification).  Every case runs pack
(unless the topology is formed inside), verify and commit through the C ABI
and is compared with the fp64 oracle: per tensor, per (request, head) and per
node row for O and U, per (request, head) for the committed state, log P to
an absolute bound, the packed topology bit for bit.  Each case is small, so
the sweep spans many combinations of kernel boundaries (32, 64 and 128 nodes,
depth 15) rather than a few large batches."""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_local_parity, rel_fro, state_unit_errors
from gated_deltanet_verification_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}
N_CASES = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_verification_gb300 import build
    build.build()


def _case(seed):
    """Shape, sizes, dtype and flags of sweep case `seed` (drawn, not listed)."""
    rng = np.random.default_rng(seed)
    shape = ["random", "random", "chain", "star", "4ary"][int(rng.integers(5))]
    dtype = "f32" if rng.random() < 0.35 else "bf16"
    # tree-size regime: small (value tiles / one CTA), up to 64, up to 128 nodes
    cap = [32, 64, 128][int(rng.integers(3))]
    if dtype == "f32":
        cap = 32 if rng.random() < 0.7 else cap  # mostly the fp32 tensor-core envelope
    B = int(rng.integers(1, 6))
    sizes = [int(rng.integers(0, cap + 1)) for _ in range(B)]
    if max(sizes) == 0:
        sizes[0] = 1
    H = int(rng.integers(1, 5))
    if shape == "chain":
        max_depth = max(sizes) - 1 if rng.random() < 0.5 else min(15, max(sizes) - 1)
        if max_depth < max(sizes) - 1:  # chains deeper than the bound are refused
            sizes = [min(s, max_depth + 1) for s in sizes]
    elif shape == "random":
        max_depth = int(rng.integers(1, 16)) if rng.random() < 0.7 else int(rng.integers(16, 60))
    else:
        max_depth = 3
    max_depth = max(max_depth, 1)
    flag = ["default", "value_tiles", "one_tile", "inline"][int(rng.integers(4))]
    return shape, dtype, B, H, sizes, max_depth, flag


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_forest_sweep(seed):
    from gated_deltanet_verification_gb300 import bole, device
    shape, dtype, B, H, sizes, max_depth, flag = _case(seed)
    b = I.random_batch(seed=9000 + seed, B=B, H=H, dk=128, dv=128, sizes=sizes,
                       max_depth=max_depth, dtype=dtype, sigma=0.05, accept="uniform",
                       shape=shape)
    f = {"default": 0, "value_tiles": bole.FLAG_VALUE_TILES,
         "one_tile": bole.FLAG_ONE_TILE_PER_HEAD, "inline": 0}[flag]
    db = device.to_device(b)
    if flag == "inline" and device.inline_topology_supported(db, f):
        f |= bole.FLAG_INLINE_TOPOLOGY
    rb = device.alloc_round(db, f)
    if f & bole.FLAG_INLINE_TOPOLOGY:
        device.verify(db, rb, f)
    else:
        device.pack(db, rb)
        device.verify(db, rb, f)
    O = rb.O.float().cpu().numpy().astype(np.float64)
    U = rb.U.cpu().numpy().astype(np.float64)
    logP = rb.logP.cpu().numpy().astype(np.float64)
    device.commit(db, rb, f & ~bole.FLAG_INLINE_TOPOLOGY)
    S_new = db.S.cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    bole.check_status(rb.status, f"sweep case {seed}")
    name = f"sweep{seed}[{shape},{dtype},B={B},H={H},sizes={sizes},d<={max_depth},{flag}]"
    if not f & bole.FLAG_INLINE_TOPOLOGY:
        depth, anc, req, st = oracle.pack(b.offsets, b.parent, b.max_depth)
        assert st == oracle.OK
        assert np.array_equal(rb.depth.cpu().numpy(), depth), name
        assert np.array_equal(rb.anc.cpu().numpy().view(np.uint32), anc), name
        assert np.array_equal(rb.req_depth[:b.B].cpu().numpy(), req), name
    Oe, Ue, Le = oracle.verify(b)
    Se = oracle.commit(b)
    tol = TOL[dtype]
    assert rel_fro(O, Oe) <= tol and rel_fro(U, Ue) <= tol, name
    assert_local_parity(name, "O", O, Oe, b.offsets, tol)
    assert_local_parity(name, "U", U, Ue, b.offsets, tol)
    assert np.max(np.abs(logP - Le)) < 2e-4 * max(1.0, np.max(np.abs(Le))), name
    assert max(state_unit_errors(S_new, Se).values()) <= tol, name


N_FUSED = 24


def _fused_case(seed):
    """Two rounds of one random workload for the deferred commit: shapes,
    request and head counts, tree sizes from empty to 64 nodes, depths up to
    15 (accepted paths of up to 16 nodes: one or two product chunks)."""
    rng = np.random.default_rng(50_000 + seed)
    B = int(rng.integers(1, 6))
    H = int(rng.integers(1, 5))
    rounds = []
    for _ in range(2):
        shape = ["random", "random", "chain", "star", "4ary"][int(rng.integers(5))]
        cap = [32, 64][int(rng.integers(2))]
        sizes = [int(rng.integers(0, cap + 1)) for _ in range(B)]
        if max(sizes) == 0:
            sizes[0] = 1
        if shape == "chain":
            sizes = [min(s, 16) for s in sizes]
            max_depth = max(max(sizes) - 1, 1)
        elif shape == "random":
            max_depth = int(rng.integers(1, 16))
        else:
            max_depth = 3
        accept = ["uniform", "deepest", "leaf"][int(rng.integers(3))]
        rounds.append((shape, sizes, max_depth, accept))
    return B, H, rounds


@pytest.mark.parametrize("seed", range(N_FUSED))
def test_commit_verify_sweep(seed):
    """bole_commit_verify on random pairs of rounds against the oracle's commit
    of the first round followed by its verification of the second."""
    import copy
    from gated_deltanet_verification_gb300 import bole, device
    B, H, rounds = _fused_case(seed)
    batches = [I.random_batch(seed=60_000 + 2 * seed + i, B=B, H=H, dk=128, dv=128, sizes=sz,
                              max_depth=md, dtype="bf16", sigma=0.05, accept=acc, shape=sh)
               for i, (sh, sz, md, acc) in enumerate(rounds)]
    prev, cur = batches
    dp, dc = device.to_device(prev), device.to_device(cur)
    st = bole.new_status()
    _, U0, L0 = bole.tree_verify(dp.S, dp.q, dp.k, dp.v, dp.gamma, dp.beta, dp.offsets, dp.parent,
                                 None, None, None, dp.max_T, dp.max_depth, status=st,
                                 flags=bole.FLAG_INLINE_TOPOLOGY)
    S = dp.S.clone()
    O, U, logP = bole.commit_verify(S, dp.k, U0, L0, dp.offsets, dp.parent, dp.accepted, dc.q,
                                    dc.k, dc.v, dc.gamma, dc.beta, dc.offsets, dc.parent,
                                    dc.max_T, dc.max_depth, status=st)
    torch.cuda.synchronize()
    bole.check_status(st, f"fused sweep case {seed}")
    S1 = oracle.commit(prev)
    cb = copy.copy(cur)
    cb.S_pre = S1
    O_ref, U_ref, lp_ref = oracle.verify(cb)
    tol = TOL["bf16"]
    name = f"fused sweep {seed} (B={B}, H={H}, rounds {rounds})"
    su = state_unit_errors(S.cpu().numpy(), S1)
    assert max(su.values()) <= tol, f"{name}: committed state worst head {max(su.values()):.3e}"
    O = O.float().cpu().numpy().astype(np.float64)
    U = U.cpu().numpy().astype(np.float64)
    assert rel_fro(O, O_ref) <= tol and rel_fro(U, U_ref) <= tol, name
    assert_local_parity(name, "O", O, O_ref, cur.offsets, tol)
    assert_local_parity(name, "U", U, U_ref, cur.offsets, tol)
    lp = logP.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lp - lp_ref), initial=0.0) < \
        2e-4 * max(1.0, np.max(np.abs(lp_ref), initial=0.0)), name
