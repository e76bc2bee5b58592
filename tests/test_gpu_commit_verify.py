"""bole_commit_verify: the previous round's commit (Eq. (10)) applied to each
head's state inside the next round's verification, so one state read serves
both.  Checked two ways:
  - against the fp64 oracle: the previous round's accepted path replayed node
    by node (the sequential recurrence), then this round's tree executed node
    by node from that committed state -- per tensor, per (request, head) and
    per node row;
  - against the library's own two-call sequence (bole_commit, then
    bole_tree_verify with the topology formed in the kernel), which it must
    reproduce bit for bit: the same products in the same order.
Edge cases: requests with no accepted node, empty and refused trees in the
new round (still committed), accepted paths of one and two eight-node product
chunks (up to the 16-node limit), faulty commit inputs (reported, that request
left uncommitted), and several rounds in a row."""
import copy

import numpy as np
import pytest
import torch

import oracle
from conftest import assert_local_parity, rel_fro, state_unit_errors
from gated_deltanet_verification_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = 1e-2  # bf16 q/k/v with fp32 state


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_verification_gb300 import build
    build.build()


def _verify(bole, db, S, status):
    """This round's verification by the one-CTA-per-head kernel (the kernel the
    fused call extends), its topology formed in the kernel."""
    return bole.tree_verify(S, db.q, db.k, db.v, db.gamma, db.beta, db.offsets, db.parent, None,
                            None, None, db.max_T, db.max_depth, status=status,
                            flags=bole.FLAG_INLINE_TOPOLOGY | bole.FLAG_ONE_TILE_PER_HEAD)


def _both(prev, cur, accepted=None, S0=None, U0L0=None):
    """The previous round verified by the two-call path (its U, logP are the
    factors both sides commit), then this round by bole_commit_verify and by
    bole_commit + bole_tree_verify from copies of the same state."""
    from gated_deltanet_verification_gb300 import bole, device
    dp, dc = device.to_device(prev), device.to_device(cur)
    acc = dp.accepted if accepted is None else torch.as_tensor(
        np.asarray(accepted, np.int32), device="cuda")
    S_in = dp.S if S0 is None else S0
    if U0L0 is None:
        st = bole.new_status()
        _, U0, L0 = _verify(bole, dp, S_in, st)
        bole.check_status(st, "previous round")
    else:
        U0, L0 = U0L0
    S_f = S_in.clone()
    st_f = bole.new_status()
    O_f, U_f, L_f = bole.commit_verify(S_f, dp.k, U0, L0, dp.offsets, dp.parent, acc, dc.q, dc.k,
                                       dc.v, dc.gamma, dc.beta, dc.offsets, dc.parent, dc.max_T,
                                       dc.max_depth, status=st_f)
    S_s = S_in.clone()
    st_s = bole.new_status()
    bole.commit(S_s, dp.k, U0, L0, dp.offsets, dp.parent, acc, status=st_s)
    O_s, U_s, L_s = _verify(bole, dc, S_s, st_s)
    torch.cuda.synchronize()
    return dict(S_f=S_f, O_f=O_f, U_f=U_f, L_f=L_f, st_f=st_f, S_s=S_s, O_s=O_s, U_s=U_s,
                L_s=L_s, st_s=st_s, acc=acc.cpu().numpy())


def _same(r, cur):
    """Bit-identical to the two-call sequence (outputs on this round's nodes)."""
    assert torch.equal(r["S_f"], r["S_s"]), "committed state differs from bole_commit"
    n = cur.N
    for a, b in (("O_f", "O_s"), ("U_f", "U_s"), ("L_f", "L_s")):
        assert torch.equal(r[a][:n], r[b][:n]), f"{a} differs from bole_tree_verify"


def _against_oracle(prev, cur, r, name):
    pb = copy.copy(prev)
    pb.accepted = r["acc"]
    S1 = oracle.commit(pb)
    su = state_unit_errors(r["S_f"].cpu().numpy(), S1)
    (wb, wh), worst = max(su.items(), key=lambda kv: kv[1])
    assert worst <= TOL, f"{name}: committed state worst (request, head) ({wb}, {wh}) {worst:.3e}"
    cb = copy.copy(cur)
    cb.S_pre = S1
    O, U, logP = oracle.verify(cb)
    got_O = r["O_f"].float().cpu().numpy()
    got_U = r["U_f"].cpu().numpy()
    assert rel_fro(got_O, O) <= TOL and rel_fro(got_U, U) <= TOL
    assert_local_parity(name, "O", got_O, O, cur.offsets, TOL)
    assert_local_parity(name, "U", got_U, U, cur.offsets, TOL)
    assert np.max(np.abs(r["L_f"].cpu().numpy() - logP), initial=0.0) < \
        2e-4 * max(1.0, np.max(np.abs(logP), initial=0.0))
    return worst


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_commit_verify_configs(cfg):
    from gated_deltanet_verification_gb300 import bole
    prev = I.config_batch(cfg, seed=1000 + cfg)
    cur = I.config_batch(cfg, seed=2000 + cfg)
    r = _both(prev, cur)
    bole.check_status(r["st_f"], "commit_verify")
    bole.check_status(r["st_s"], "commit + verify")
    _same(r, cur)
    worst = _against_oracle(prev, cur, r, f"config {cfg}")
    print(f"config {cfg}: committed state worst head {worst:.2e}")


@pytest.mark.parametrize("layout_T", [32, 64])
def test_commit_verify_edges(layout_T):
    """Paths of 1, 16 (the limit: two product chunks), 9 and 12 nodes, a
    request without an accepted node and one whose previous tree was empty;
    the new round has empty, one-node and full trees (both tree layouts)."""
    from gated_deltanet_verification_gb300 import bole
    prev = I.random_batch(seed=31, B=6, H=3, dk=128, dv=128, sizes=[1, 16, 9, 0, 12, 5],
                          max_depth=15, dtype="bf16", sigma=0.05, accept="deepest", shape="chain")
    cur_sizes = [3, 0, layout_T, 8, 1, layout_T // 2]
    cur = I.random_batch(seed=32, B=6, H=3, dk=128, dv=128, sizes=cur_sizes, max_depth=6,
                         dtype="bf16", sigma=0.05)
    acc = prev.accepted.copy()
    acc[4] = -1  # no commit for request 4
    r = _both(prev, cur, accepted=acc)
    bole.check_status(r["st_f"], "commit_verify")
    _same(r, cur)
    _against_oracle(prev, cur, r, f"edges T<={layout_T}")
    # request 4's state is untouched, request 3 (empty previous tree) too
    S0 = torch.as_tensor(prev.S_pre, device="cuda")
    assert torch.equal(r["S_f"][4], S0[4]) and torch.equal(r["S_f"][3], S0[3])


def test_commit_verify_commits_refused_trees():
    """A new tree deeper than max_depth is refused (BOLE_ERR_DEPTH, no outputs
    for it) while every request's previous round is still committed."""
    from gated_deltanet_verification_gb300 import bole, device
    prev = I.random_batch(seed=41, B=3, H=2, dk=128, dv=128, sizes=[6, 10, 4], max_depth=15,
                          dtype="bf16", sigma=0.05, accept="deepest", shape="chain")
    cur = I.random_batch(seed=42, B=3, H=2, dk=128, dv=128, sizes=[5, 12, 7], max_depth=15,
                         dtype="bf16", sigma=0.05, shape="chain")
    cur.max_depth = 6  # request 1's 12-node chain (depth 11) is refused, the others pass
    r = _both(prev, cur)
    code = int(r["st_f"][0].item())
    assert code == bole.ERR_DEPTH
    pb = copy.copy(prev)
    S1 = oracle.commit(pb)
    su = state_unit_errors(r["S_f"].cpu().numpy(), S1)
    assert max(su.values()) <= TOL


def test_commit_verify_rejects_faulty_commit_inputs():
    """A previous path over 16 nodes (BOLE_ERR_DEPTH {request, node, 16}) and
    an accepted node past its tree (BOLE_ERR_BAD_TOPOLOGY): that request's
    state is left uncommitted, the other requests are committed and verified."""
    from gated_deltanet_verification_gb300 import bole, device
    prev = I.random_batch(seed=51, B=2, H=2, dk=128, dv=128, sizes=[20, 5], max_depth=19,
                          dtype="bf16", sigma=0.05, accept="deepest", shape="chain")
    cur = I.random_batch(seed=52, B=2, H=2, dk=128, dv=128, sizes=[6, 6], max_depth=5,
                         dtype="bf16", sigma=0.05)
    dp = device.to_device(prev)
    S0 = dp.S.clone()
    rb = device.alloc_round(dp)  # a 20-node chain: the large-tree kernel, after pack
    device.pack(dp, rb)
    device.verify(dp, rb, 0)
    bole.check_status(rb.status, "previous round")
    U0, L0 = rb.U, rb.logP
    r = _both(prev, cur, S0=S0, U0L0=(U0, L0))
    s = r["st_f"].cpu().numpy()
    assert s[0] == bole.ERR_DEPTH and s[1] == 0 and s[2] == int(prev.accepted[0]) and s[3] == 16
    assert torch.equal(r["S_f"][0], S0[0])  # not committed
    # request 1 is committed and verified as by the two calls
    assert torch.equal(r["S_f"][1], r["S_s"][1])
    o1, e1 = int(cur.offsets[1]), int(cur.offsets[2])
    assert torch.equal(r["O_f"][o1:e1], r["O_s"][o1:e1])
    # an accepted node past its tree
    r = _both(prev, cur, accepted=[int(prev.tree_sizes()[0]) + 3, 2], S0=S0, U0L0=(U0, L0))
    s = r["st_f"].cpu().numpy()
    assert s[0] == bole.ERR_BAD_TOPOLOGY and s[1] == 0
    assert torch.equal(r["S_f"][0], S0[0])


def test_commit_verify_rounds():
    """Four rounds in a row, each committing the one before: the fused
    sequence matches the two-call sequence bit for bit at every round."""
    from gated_deltanet_verification_gb300 import bole, device
    rounds = [I.random_batch(seed=60 + i, B=4, H=4, dk=128, dv=128, sizes=[9, 17, 32, 4],
                             max_depth=8, dtype="bf16", sigma=0.05, accept="uniform")
              for i in range(4)]
    db = [device.to_device(b) for b in rounds]
    S_f = db[0].S.clone()
    S_s = db[0].S.clone()
    st = bole.new_status()
    O_f, U_f, L_f = _verify(bole, db[0], S_f, st)
    O_s, U_s, L_s = _verify(bole, db[0], S_s, st)
    for i in range(1, 4):
        p, c = db[i - 1], db[i]
        O_f, U_f2, L_f2 = bole.commit_verify(S_f, p.k, U_f, L_f, p.offsets, p.parent, p.accepted,
                                             c.q, c.k, c.v, c.gamma, c.beta, c.offsets, c.parent,
                                             c.max_T, c.max_depth, status=st)
        bole.commit(S_s, p.k, U_s, L_s, p.offsets, p.parent, p.accepted, status=st)
        O_s, U_s, L_s = _verify(bole, c, S_s, st)
        U_f, L_f = U_f2, L_f2
        torch.cuda.synchronize()
        bole.check_status(st, f"round {i}")
        assert torch.equal(S_f, S_s) and torch.equal(O_f, O_s) and torch.equal(U_f, U_s)
