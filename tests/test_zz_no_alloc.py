"""bole_tree_verify_noalloc: the verification entry point that allocates
nothing, for callers that cannot allocate device memory when they verify
(hosts that hand over only their own tensors, serving loops that forbid
allocation on the hot path).  Its G, C scratch is a fixed library-owned
array; these tests call it through the C ABI and compare it with
bole_tree_verify (same CUDA-core kernels, caller-allocated workspace) and with
the fp64 CPU oracle, on two calls in a row of different sizes, so stale
scratch from the first call must not leak into the second.  Collected last on
purpose."""
import numpy as np
import pytest
import torch

import oracle
from conftest import assert_local_parity, rel_fro
from gated_deltanet_verification_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_verification_gb300 import build
    build.build()


def _both(batch):
    from gated_deltanet_verification_gb300 import bole, device
    db = device.to_device(batch)
    rb = device.alloc_round(db, bole.FLAG_FORCE_SIMT)
    device.pack(db, rb)
    device.verify(db, rb, bole.FLAG_FORCE_SIMT)
    ref = [t.float().cpu().numpy() for t in (rb.O, rb.U, rb.logP)]
    st = bole.new_status()
    st.copy_(rb.status)
    O2, U2, L2 = bole.tree_verify_noalloc(
        db.S, db.q, db.k, db.v, db.gamma, db.beta, db.offsets, db.parent, rb.depth, rb.anc,
        rb.req_depth[:db.B], db.max_T, db.max_depth, status=st)
    torch.cuda.synchronize()
    bole.check_status(st, "noalloc verify")
    got = [t.float().cpu().numpy() for t in (O2, U2, L2)]
    return ref, got


def test_noalloc_matches_workspace_path_two_calls():
    first = I.config_batch(2)                       # 16 x 32 heads, 32-node trees (bf16)
    second = I.random_batch(seed=11, B=5, H=3, dk=64, dv=48, sizes=[17, 9, 1, 30, 12],
                            max_depth=6, dtype="f32", sigma=0.1)
    for batch in (first, second):
        ref, got = _both(batch)
        for r, g in zip(ref, got):
            assert rel_fro(g, r) <= TOL[batch.dtype]
        # and against the oracle, so an error the two CUDA-core runs share
        # cannot pass: O and U per tensor, per (request, head) and per node row
        O, U, logP = oracle.verify(batch)
        tol = TOL[batch.dtype]
        assert rel_fro(got[0], O) <= tol and rel_fro(got[1], U) <= tol
        assert_local_parity(batch.name, "O", got[0], O, batch.offsets, tol)
        assert_local_parity(batch.name, "U", got[1], U, batch.offsets, tol)
        assert np.max(np.abs(got[2] - logP)) < 2e-4 * max(1.0, np.max(np.abs(logP)))


def test_noalloc_rejects_oversize():
    from gated_deltanet_verification_gb300 import bole, device
    b = I.random_batch(seed=3, B=2, H=2, dk=16, dv=16, sizes=[4, 4], max_depth=3)
    db = device.to_device(b)
    rb = device.alloc_round(db)
    device.pack(db, rb)
    # declare trees of up to 128 nodes over enough heads to exceed the array
    big_B, big_H = 64, 2
    assert big_B * big_H * 128 * 128 > bole.NOALLOC_MAX_FACTOR_ELEMS
    offsets = torch.zeros(big_B + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(bole.BoleError) as e:
        bole.tree_verify_noalloc(db.S, db.q[:, :1].repeat(1, big_H, 1).contiguous(),
                                 db.k[:, :1].repeat(1, big_H, 1).contiguous(),
                                 db.v[:, :1].repeat(1, big_H, 1).contiguous(),
                                 db.gamma[:, :1].repeat(1, big_H).contiguous(),
                                 db.beta[:, :1].repeat(1, big_H).contiguous(), offsets,
                                 db.parent, rb.depth, rb.anc,
                                 torch.zeros(big_B, dtype=torch.int32, device="cuda"), 128, 3)
    assert e.value.code == bole.ERR_UNSUPPORTED
