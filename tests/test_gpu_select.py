"""GPU parity for the device-side proposal selection and forest build against
the oracle in oracle/select.py: every output is an integer decision taken on
float32 scores both sides accumulate root-down, so the scores must agree bit
for bit and the forest (offsets, local parents, candidate map) exactly."""
import numpy as np
import pytest
import torch

import oracle
from conftest import rel_fro
from gated_deltanet_verification_gb300 import inputs as I
from oracle import select as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_verification_gb300 import build
    build.build()


def _t(a, dt=torch.int32):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dt)


def _gpu(d, budget, caps="given"):
    from gated_deltanet_verification_gb300 import bole
    cp = None if caps is None else _t(d.caps if caps == "given" else caps)
    off, par, src, rho, st = bole.select_forest(_t(d.p, torch.float32), _t(d.cand_offsets),
                                                _t(d.cand_parent), budget, caps=cp)
    torch.cuda.synchronize()
    return (off.cpu().numpy(), par.cpu().numpy(), src.cpu().numpy(), rho.cpu().numpy(),
            st.cpu().tolist())


def _check(d, budget, caps="given"):
    got_off, got_par, got_src, got_rho, st = _gpu(d, budget, caps)
    assert st[0] == 0, st
    c = None if caps is None else (d.caps if caps == "given" else caps)
    off, par, src, rho = S.select_forest(d.p, d.cand_offsets, d.cand_parent, budget, c)
    assert np.array_equal(got_rho[:d.M].view(np.uint32), rho.view(np.uint32))
    assert np.array_equal(got_off, off), (got_off, off)
    n = int(off[-1])
    assert np.array_equal(got_par[:n], par)
    assert np.array_equal(got_src[:n], src)
    return n


@pytest.mark.parametrize("seed,B,m,depth", [(1, 4, (10, 30), 6), (2, 64, (64, 256), 12),
                                            (3, 17, (1, 200), 9), (4, 200, (50, 300), 8)])
def test_selection_matches_oracle(seed, B, m, depth):
    d = I.draft_candidates(seed, B, m[0], m[1], depth)
    total = int(np.minimum(np.diff(d.cand_offsets), d.caps).sum())
    for budget in (0, 1, B - 1, B, 3 * B, 2048, total, total + 100):
        if budget >= 0:
            _check(d, budget)


def test_no_caps_and_large_requests():
    d = I.draft_candidates(5, 6, 900, 1024, 30, max_children=2)
    for budget in (6, 300, 10 ** 5):
        n = _check(d, budget, caps=None)
        assert n <= 6 * 128


def test_deep_chains_and_ties():
    B, M = 3, 1024
    offs = np.arange(B + 1, dtype=np.int32) * M
    par = np.tile(np.arange(-1, M - 1, dtype=np.int32), B)
    d = I.DraftCandidates(offs, par, np.ones(B * M, np.float32), np.array([5, 128, 1], np.int32))
    _check(d, 100)  # every score ties at 1: depth, then request, then index
    d.p[:] = np.float32(0.999)
    _check(d, 100)
    _check(d, 1000, caps=None)


def test_bad_candidate_link_is_reported():
    d = I.draft_candidates(7, 5, 10, 20, 4)
    d.cand_parent[d.cand_offsets[2] + 3] = 5  # a forward link in request 2
    off, par, src, rho, st = _gpu(d, 40)
    assert st[:3] == [3, 2, int(d.cand_offsets[2]) + 3]
    assert off[3] - off[2] == 0  # that request receives no nodes


def test_selected_forest_feeds_pack_and_verify_without_host_round_trip():
    """select -> pack (N = the budget capacity) -> verify on the candidates'
    operands gathered by src, against the oracle on the compacted batch."""
    from gated_deltanet_verification_gb300 import bole
    d = I.draft_candidates(11, 16, 40, 120, 8)
    budget = 400
    H, dk, dv = 4, 128, 128
    rng = np.random.default_rng(3)
    qc = I.round_to_bf16(rng.standard_normal((d.M, H, dk)).astype(np.float32) / np.sqrt(dk))
    kc = I.round_to_bf16(rng.standard_normal((d.M, H, dk)).astype(np.float32) / np.sqrt(dk))
    vc = I.round_to_bf16(rng.standard_normal((d.M, H, dv)).astype(np.float32))
    gc = np.exp(-np.logaddexp(0, rng.standard_normal((d.M, H)))).astype(np.float32)
    bc = (1 / (1 + np.exp(-rng.standard_normal((d.M, H))))).astype(np.float32)
    S_pre = (0.05 * rng.standard_normal((d.B, H, dk, dv))).astype(np.float32)

    # src past the node count stays 0 (a valid gather index)
    src0 = torch.zeros(budget, dtype=torch.int32, device="cuda")
    off, par, src, _, st = bole.select_forest(_t(d.p, torch.float32), _t(d.cand_offsets),
                                              _t(d.cand_parent), budget, caps=_t(d.caps),
                                              src=src0)
    status = bole.new_status()
    depth, anc, req, _ = bole.pack_forest(off, par, 127, status=status)
    idx = src.long()
    q, k, v = (_t(x, torch.bfloat16)[idx] for x in (qc, kc, vc))
    g, bt = (_t(x, torch.float32)[idx] for x in (gc, bc))
    O, U, logP = bole.tree_verify(_t(S_pre, torch.float32), q, k, v, g, bt, off, par, depth,
                                  anc, req, 64, 15, status=status)
    torch.cuda.synchronize()
    assert st.cpu().tolist()[0] == 0
    bole.check_status(status)
    eo, ep, es, _ = S.select_forest(d.p, d.cand_offsets, d.cand_parent, budget, d.caps)
    n = int(eo[-1])
    b = I.TreeBatch("selected", d.B, H, dk, dv, "bf16", 127, eo, ep, qc[es], kc[es], vc[es],
                    gc[es], bc[es], S_pre, np.full(d.B, -1, np.int32))
    Oe, Ue, _ = oracle.verify(b)
    assert rel_fro(O[:n].float().cpu().numpy(), Oe) <= 1e-2
    assert rel_fro(U[:n].cpu().numpy(), Ue) <= 1e-2


def test_empty_batch_gives_the_empty_forest():
    from gated_deltanet_verification_gb300 import bole
    off = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    o, _, _, _, st = bole.select_forest(torch.zeros(1, dtype=torch.float32, device="cuda"),
                                        torch.zeros(1, dtype=torch.int32, device="cuda"),
                                        torch.zeros(1, dtype=torch.int32, device="cuda"), 10,
                                        offsets=off)
    torch.cuda.synchronize()
    assert o.cpu().tolist() == [0] and st.cpu().tolist()[0] == 0
