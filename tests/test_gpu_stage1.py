"""GPU parity for stage 1 (tree-parallel causal convolution + gates) and the
convolution-state commit, against the float64 oracle in oracle/stage1.py on
the same seeded inputs.  q, k, v within relative Frobenius 1e-2 (bf16
outputs) or 1e-5 (float32); gamma and beta (float32) within 1e-5 relative
per element; the committed convolution state bit for bit (rows are copied)."""
import numpy as np
import pytest
import torch

import oracle
from conftest import rel_fro
from gated_deltanet_verification_gb300 import inputs as I
from oracle import stage1

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_verification_gb300 import build
    build.build()


def _t(a, dt):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dt)


def _xdt(s):
    return torch.bfloat16 if s.dtype == "bf16" else torch.float32


def _gpu_stage1(batch, s, status=None):
    from gated_deltanet_verification_gb300 import bole
    dt = _xdt(s)
    st = bole.new_status() if status is None else status
    out = bole.conv_gates(
        _t(s.x, dt), _t(s.conv_state, dt) if s.W > 1 else None, _t(s.conv_w, torch.float32),
        _t(s.conv_b, torch.float32), _t(s.a, torch.float32), _t(s.b, torch.float32),
        _t(batch.offsets, torch.int32), _t(batch.parent, torch.int32), batch.H, batch.dk,
        batch.dv, max(batch.max_T, 1),
        gate_scale=None if s.gate_scale is None else _t(s.gate_scale, torch.float32),
        gate_bias=None if s.gate_bias is None else _t(s.gate_bias, torch.float32), status=st)
    torch.cuda.synchronize()
    return [o.float().cpu().numpy().astype(np.float64) for o in out], st


def _oracle_stage1(batch, s):
    return stage1.conv_gates(s.x, s.conv_state, s.conv_w, s.conv_b, s.a, s.b, batch.offsets,
                             batch.parent, batch.H, batch.dk, batch.dv, s.gate_scale,
                             s.gate_bias)


CASES = [
    ("cfg2-w4", lambda: I.config_batch(2), 4, None, False),
    ("cfg3-w4", lambda: I.config_batch(3), 4, None, True),
    ("chain128-w4", lambda: I.config_batch(4, shape="chain"), 4, None, False),
    ("star128-w8", lambda: I.config_batch(4, shape="star"), 8, None, False),
    ("ragged-w1", lambda: I.random_batch(seed=90, B=5, H=3, dk=128, dv=128,
                                         sizes=[9, 0, 64, 1, 33], max_depth=12, dtype="bf16"),
     1, None, True),
    ("f32-w3", lambda: I.random_batch(seed=91, B=4, H=2, dk=32, dv=48, sizes=[17, 5, 0, 30],
                                      max_depth=6, dtype="f32"), 3, "f32", True),
    ("f32-small-w2", lambda: I.random_batch(seed=92, B=2, H=5, dk=16, dv=16, sizes=[8, 3],
                                            max_depth=3, dtype="f32"), 2, "f32", False),
]


@pytest.mark.parametrize("name,make,W,dtype,gate_terms", CASES, ids=[c[0] for c in CASES])
def test_conv_gates_parity(name, make, W, dtype, gate_terms):
    from gated_deltanet_verification_gb300 import bole
    b = make()
    s = I.stage1_inputs(b, W=W, seed=11, dtype=dtype, gate_terms=gate_terms)
    (q, k, v, g, bt), st = _gpu_stage1(b, s)
    bole.check_status(st)
    qe, ke, ve, ge, bte = _oracle_stage1(b, s)
    tol = TOL[s.dtype]
    for nm, x, e in (("q", q, qe), ("k", k, ke), ("v", v, ve)):
        assert rel_fro(x, e) <= tol, (nm, rel_fro(x, e))
    assert np.max(np.abs(g - ge) / ge) <= 1e-5
    assert np.max(np.abs(bt - bte) / bte) <= 1e-5
    # q, k leave as unit vectors per head (up to output rounding)
    nq = np.linalg.norm(q, axis=-1)
    assert np.max(np.abs(nq - 1)) <= (1e-2 if s.dtype == "bf16" else 1e-5)


@pytest.mark.parametrize("W", [2, 4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_conv_commit_bit_exact(W, dtype):
    from gated_deltanet_verification_gb300 import bole
    b = I.random_batch(seed=93 + W, B=6, H=2, dk=32, dv=16, sizes=[12, 1, 0, 40, 7, 128],
                       max_depth=127, dtype="f32", accept="uniform", shape="chain")
    b.accepted[3] = -1
    s = I.stage1_inputs(b, W=W, seed=3, dtype=dtype)
    dt = _xdt(s)
    st_dev = _t(s.conv_state, dt)
    status = bole.new_status()
    bole.conv_commit(st_dev, _t(s.x, dt), _t(b.offsets, torch.int32),
                     _t(b.parent, torch.int32), _t(b.accepted, torch.int32), status=status)
    torch.cuda.synchronize()
    bole.check_status(status)
    exp = stage1.conv_commit(s.conv_state, s.x, b.offsets, b.parent, b.accepted)
    assert np.array_equal(st_dev.float().cpu().numpy(), exp)


def test_conv_commit_on_random_trees_bit_exact():
    from gated_deltanet_verification_gb300 import bole
    b = I.config_batch(3)
    s = I.stage1_inputs(b, W=4, seed=5)
    st_dev = _t(s.conv_state, torch.bfloat16)
    bole.conv_commit(st_dev, _t(s.x, torch.bfloat16), _t(b.offsets, torch.int32),
                     _t(b.parent, torch.int32), _t(b.accepted, torch.int32))
    torch.cuda.synchronize()
    exp = stage1.conv_commit(s.conv_state, s.x, b.offsets, b.parent, b.accepted)
    assert np.array_equal(st_dev.float().cpu().numpy(), exp)


def test_bad_parent_link_is_reported_and_request_left_unwritten():
    from gated_deltanet_verification_gb300 import bole
    b = I.random_batch(seed=94, B=3, H=2, dk=16, dv=16, sizes=[5, 6, 4], max_depth=4,
                       dtype="f32")
    b.parent[b.offsets[1] + 3] = 4          # a forward link in request 1
    s = I.stage1_inputs(b, W=4, seed=1)
    (q, k, v, g, bt), st = _gpu_stage1(b, s)
    code, req, node, detail = st.cpu().tolist()
    assert (code, req, node, detail) == (bole.ERR_BAD_TOPOLOGY, 1, int(b.offsets[1]) + 3, 4)


def test_full_layer_round_matches_oracle_chain():
    """stage 1 -> pack -> verify -> commit (and the conv-state commit) on
    device, against oracle stage 1 -> verify -> commit on the bf16-rounded
    operands."""
    from gated_deltanet_verification_gb300 import bole
    b = I.config_batch(2)
    s = I.stage1_inputs(b, W=4, seed=21)
    dt = torch.bfloat16
    offsets, parent = _t(b.offsets, torch.int32), _t(b.parent, torch.int32)
    x = _t(s.x, dt)
    status = bole.new_status()
    depth, anc, req, _ = bole.pack_forest(offsets, parent, b.max_depth, status=status)
    q, k, v, g, bt = bole.conv_gates(x, _t(s.conv_state, dt), _t(s.conv_w, torch.float32),
                                     _t(s.conv_b, torch.float32), _t(s.a, torch.float32),
                                     _t(s.b, torch.float32), offsets, parent, b.H, b.dk, b.dv,
                                     b.max_T, status=status)
    S = _t(b.S_pre, torch.float32)
    O, U, logP = bole.tree_verify(S, q, k, v, g, bt, offsets, parent, depth, anc, req,
                                  b.max_T, b.max_depth, status=status)
    acc = _t(b.accepted, torch.int32)
    bole.commit(S, k, U, logP, offsets, parent, acc, status=status)
    cs = _t(s.conv_state, dt)
    bole.conv_commit(cs, x, offsets, parent, acc, status=status)
    torch.cuda.synchronize()
    bole.check_status(status)
    # oracle chain on the same inputs
    qe, ke, ve, ge, bte = _oracle_stage1(b, s)
    ob = I.TreeBatch(b.name, b.B, b.H, b.dk, b.dv, "bf16", b.max_depth, b.offsets, b.parent,
                     I.round_to_bf16(qe.astype(np.float32)),
                     I.round_to_bf16(ke.astype(np.float32)),
                     I.round_to_bf16(ve.astype(np.float32)), ge.astype(np.float32),
                     bte.astype(np.float32), b.S_pre, b.accepted)
    Oe, Ue, _ = oracle.verify(ob)
    Se = oracle.commit(ob)
    assert rel_fro(O.float().cpu().numpy(), Oe) <= TOL["bf16"]
    assert rel_fro(U.cpu().numpy(), Ue) <= TOL["bf16"]
    assert rel_fro(S.cpu().numpy(), Se) <= TOL["bf16"]
    exp = stage1.conv_commit(s.conv_state, s.x, b.offsets, b.parent, b.accepted)
    assert np.array_equal(cs.float().cpu().numpy(), exp)


def test_tree_larger_than_max_T_is_reported():
    from gated_deltanet_verification_gb300 import bole
    b = I.random_batch(seed=95, B=2, H=2, dk=16, dv=16, sizes=[5, 9], max_depth=8, dtype="f32")
    s = I.stage1_inputs(b, W=4, seed=2)
    st = bole.new_status()
    bole.conv_gates(_t(s.x, torch.float32), _t(s.conv_state, torch.float32),
                    _t(s.conv_w, torch.float32), None, _t(s.a, torch.float32),
                    _t(s.b, torch.float32), _t(b.offsets, torch.int32),
                    _t(b.parent, torch.int32), b.H, b.dk, b.dv, 8, status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [bole.ERR_BAD_TOPOLOGY, 1, -1, 9]
