"""GPU parity for the state-slot layout and the unified cross-layer commit.

* BOLE_FLAG_STATE_VK: S_pre / S stored [B, H, dv, dk] (the serving runtime's
  canonical slot layout, Section IV-D).  O and U against the oracle, the
  committed slots against the oracle's commit transposed, on the fused,
  large-tree and CUDA-core kernels.
* bole_commit_layers: one launch commits several layers that verified the
  same forest (each layer's own S_pre, q, k, v, gamma, beta), their factors in
  one contiguous [layers, ...] buffer and their states in a pool with gaps.
  Every layer against the oracle, and bit for bit against that layer's own
  single-layer bole_commit.
Tolerances as in test_gpu_parity: relative Frobenius 1e-2 for bf16 q/k/v with
float32 state, 1e-5 for float32 q/k/v."""
import numpy as np
import pytest
import torch

import oracle
from conftest import rel_fro
from gated_deltanet_verification_gb300 import inputs as I

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


def _qkv_dtype(batch):
    return torch.bfloat16 if batch.dtype == "bf16" else torch.float32


def _verify_into(batch, S_pre, k, U, logP, flags):
    """pack + verify of one layer; S_pre, k, U, logP are device views the
    caller owns (slices of layered buffers).  Returns O (float64, host)."""
    from gated_deltanet_verification_gb300 import bole
    dt = _qkv_dtype(batch)
    offsets, parent = _t(batch.offsets, torch.int32), _t(batch.parent, torch.int32)
    q, v = _t(batch.q, dt), _t(batch.v, dt)
    gamma, beta = _t(batch.gamma, torch.float32), _t(batch.beta, torch.float32)
    max_T = max(batch.max_T, 1)
    depth, anc, req, st = bole.pack_forest(offsets, parent, batch.max_depth)
    O, _, _ = bole.tree_verify(S_pre, q, k, v, gamma, beta, offsets, parent, depth, anc, req,
                               max_T, batch.max_depth, U=U, logP=logP, status=st, flags=flags)
    torch.cuda.synchronize()
    bole.check_status(st)
    return O.float().cpu().numpy().astype(np.float64)


def _state(batch, layout):
    S = batch.S_pre
    return S if layout == "kv" else np.ascontiguousarray(S.transpose(0, 1, 3, 2))


CASES = [
    # (name, batch factory, extra flags)
    ("cfg2-fused", lambda: I.config_batch(2), 0),
    ("ragged-fused", lambda: I.random_batch(seed=77, B=5, H=3, dk=128, dv=128,
                                            sizes=[64, 1, 0, 37, 9], max_depth=15,
                                            dtype="bf16", sigma=0.05), 0),
    ("chain-large", lambda: I.random_batch(seed=78, B=3, H=2, dk=128, dv=128,
                                           sizes=[128, 70, 3], max_depth=127, dtype="bf16",
                                           sigma=0.05, accept="deepest", shape="chain"), 0),
    ("cfg1-simt", lambda: I.config_batch(1), 1),
    ("f32-simt", lambda: I.random_batch(seed=79, B=4, H=2, dk=32, dv=48, sizes=[9, 17, 1, 30],
                                        max_depth=9, dtype="f32", sigma=0.1), 0),
    ("f32-tc", lambda: I.random_batch(seed=83, B=4, H=3, dk=128, dv=128, sizes=[32, 9, 1, 30],
                                      max_depth=12, dtype="f32", sigma=0.1), 0),
    # fp32 keys on accepted paths of 100 and 40 nodes (the path by pointer jumping, the
    # rows in batches of eight)
    ("f32-chain", lambda: I.random_batch(seed=85, B=2, H=2, dk=128, dv=128, sizes=[100, 40],
                                         max_depth=99, dtype="f32", sigma=0.1, accept="deepest",
                                         shape="chain"), 0),
]


@pytest.mark.parametrize("name,make,extra", CASES, ids=[c[0] for c in CASES])
def test_slot_layout_verify_and_commit(name, make, extra):
    """The transposed slot layout gives the oracle's O, U and (transposed)
    committed state, and the same numbers as the default layout."""
    from gated_deltanet_verification_gb300 import bole
    b = make()
    flags = bole.FLAG_FORCE_SIMT if extra else 0
    dt = _qkv_dtype(b)
    O_ref, U_ref, _ = oracle.verify(b)
    S_ref = oracle.commit(b)
    res = {}
    for layout in ("kv", "vk"):
        f = flags | (bole.FLAG_STATE_VK if layout == "vk" else 0)
        S = _t(_state(b, layout), torch.float32)
        k = _t(b.k, dt)
        U = torch.empty((b.N, b.H, b.dv), dtype=torch.float32, device="cuda")
        logP = torch.empty((b.N, b.H), dtype=torch.float32, device="cuda")
        O = _verify_into(b, S, k, U, logP, f)
        st = bole.new_status()
        bole.commit(S, k, U, logP, _t(b.offsets, torch.int32), _t(b.parent, torch.int32),
                    _t(b.accepted, torch.int32), status=st, flags=f)
        torch.cuda.synchronize()
        bole.check_status(st)
        S_new = S.cpu().numpy().astype(np.float64)
        if layout == "vk":
            S_new = S_new.transpose(0, 1, 3, 2)
        Un = U.cpu().numpy().astype(np.float64)
        tol = TOL[b.dtype]
        assert rel_fro(O, O_ref) <= tol, (layout, rel_fro(O, O_ref))
        assert rel_fro(Un, U_ref) <= tol, (layout, rel_fro(Un, U_ref))
        assert rel_fro(S_new, S_ref) <= tol, (layout, rel_fro(S_new, S_ref))
        res[layout] = (O, Un, S_new)
    for x, y in zip(res["kv"], res["vk"]):
        assert rel_fro(y, x) <= 1e-5


LAYER_CASES = [
    ("cfg2-tc", lambda: I.config_batch(2), 0, 4),
    ("ragged-tc", lambda: I.random_batch(seed=81, B=6, H=3, dk=128, dv=128,
                                         sizes=[64, 1, 0, 37, 9, 128], max_depth=40,
                                         dtype="bf16", sigma=0.05), 0, 3),
    ("cfg2-simt", lambda: I.config_batch(2), 1, 2),
    ("f32-simt", lambda: I.random_batch(seed=82, B=4, H=2, dk=32, dv=48, sizes=[9, 17, 1, 30],
                                        max_depth=9, dtype="f32", sigma=0.1), 0, 3),
    ("f32-tc", lambda: I.random_batch(seed=84, B=4, H=3, dk=128, dv=128, sizes=[32, 9, 1, 30],
                                      max_depth=12, dtype="f32", sigma=0.1), 0, 3),
]


@pytest.mark.parametrize("layout", ["kv", "vk"])
@pytest.mark.parametrize("name,make,extra,n_layers", LAYER_CASES, ids=[c[0] for c in LAYER_CASES])
def test_commit_layers(name, make, extra, n_layers, layout):
    from gated_deltanet_verification_gb300 import bole
    base = make()
    if base.B > 1:
        base.accepted[1] = -1  # a request whose every layer stays untouched
    layers = I.layer_batches(base, n_layers, seed=123)
    flags = (bole.FLAG_FORCE_SIMT if extra else 0) | (bole.FLAG_STATE_VK if layout == "vk" else 0)
    dt = _qkv_dtype(base)
    B, H, dk, dv, N = base.B, base.H, base.dk, base.dv, base.N
    # state pool with a slot between layers: layer l at pool[2 l]
    pool0 = np.zeros((2 * n_layers,) + _state(base, layout).shape, np.float32)
    for li, lb in enumerate(layers):
        pool0[2 * li] = _state(lb, layout)
        pool0[2 * li + 1] = np.random.default_rng(li).standard_normal(pool0.shape[1:])
    pool = _t(pool0, torch.float32)
    S_layers = pool[0::2]
    k_all = torch.stack([_t(lb.k, dt) for lb in layers])
    U_all = torch.empty((n_layers, N, H, dv), dtype=torch.float32, device="cuda")
    lp_all = torch.empty((n_layers, N, H), dtype=torch.float32, device="cuda")
    for li, lb in enumerate(layers):
        _verify_into(lb, S_layers[li], k_all[li], U_all[li], lp_all[li], flags)
    # the single-layer commits on copies, for the bitwise comparison
    singles = []
    for li in range(n_layers):
        S1 = S_layers[li].clone()
        bole.commit(S1, k_all[li], U_all[li], lp_all[li], _t(base.offsets, torch.int32),
                    _t(base.parent, torch.int32), _t(base.accepted, torch.int32), flags=flags)
        singles.append(S1)
    st = bole.new_status()
    bole.commit_layers(S_layers, k_all, U_all, lp_all, _t(base.offsets, torch.int32),
                       _t(base.parent, torch.int32), _t(base.accepted, torch.int32), status=st,
                       flags=flags)
    torch.cuda.synchronize()
    bole.check_status(st)
    got = pool.cpu().numpy()
    ref = oracle.commit_layers(layers, state_layout=layout)
    for li in range(n_layers):
        e = rel_fro(got[2 * li], ref[li])
        assert e <= TOL[base.dtype], (li, e)
        assert torch.equal(S_layers[li], singles[li]), li
        assert np.array_equal(got[2 * li + 1], pool0[2 * li + 1])  # the gap slots untouched
        if base.B > 1:
            assert np.array_equal(got[2 * li][1], pool0[2 * li][1])  # accepted = -1


def test_commit_layers_reports_a_bad_accepted_node_once():
    from gated_deltanet_verification_gb300 import bole
    base = I.random_batch(seed=83, B=3, H=2, dk=128, dv=128, sizes=[10, 12, 7], max_depth=6,
                          dtype="bf16", sigma=0.05)
    layers = I.layer_batches(base, 3, seed=5)
    acc = base.accepted.copy()
    acc[2] = 7  # == tree size: out of range
    S = torch.stack([_t(lb.S_pre, torch.float32) for lb in layers])
    S0 = S.clone()
    k = torch.stack([_t(lb.k, torch.bfloat16) for lb in layers])
    U = torch.zeros((3, base.N, 2, 128), dtype=torch.float32, device="cuda")
    lp = torch.zeros((3, base.N, 2), dtype=torch.float32, device="cuda")
    st = bole.new_status()
    bole.commit_layers(S, k, U, lp, _t(base.offsets, torch.int32), _t(base.parent, torch.int32),
                       _t(acc, torch.int32), status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [bole.ERR_BAD_TOPOLOGY, 2, 7, 7]
    assert torch.equal(S[:, 2], S0[:, 2])


def test_commit_layers_overlapped_after_verify_matches_plain_launch():
    """Launched to overlap the last verification (programmatic dependent
    launch), the cross-layer commit gives bit-identical states."""
    from gated_deltanet_verification_gb300 import bole
    base = I.config_batch(2)
    layers = I.layer_batches(base, 3, seed=77)
    N, H = base.N, base.H
    out = []
    for flags in (0, bole.FLAG_OVERLAP_LAUNCH):
        S = torch.stack([_t(lb.S_pre, torch.float32) for lb in layers])
        k = torch.stack([_t(lb.k, torch.bfloat16) for lb in layers])
        U = torch.empty((3, N, H, base.dv), dtype=torch.float32, device="cuda")
        lp = torch.empty((3, N, H), dtype=torch.float32, device="cuda")
        offsets, parent = _t(base.offsets, torch.int32), _t(base.parent, torch.int32)
        depth, anc, req, st = bole.pack_forest(offsets, parent, base.max_depth)
        for li, lb in enumerate(layers):
            bole.tree_verify(S[li], _t(lb.q, torch.bfloat16), k[li], _t(lb.v, torch.bfloat16),
                             _t(lb.gamma, torch.float32), _t(lb.beta, torch.float32), offsets,
                             parent, depth, anc, req, base.max_T, base.max_depth, U=U[li],
                             logP=lp[li], status=st, flags=flags)
        bole.commit_layers(S, k, U, lp, offsets, parent, _t(base.accepted, torch.int32),
                           status=st, flags=flags)
        torch.cuda.synchronize()
        bole.check_status(st)
        out.append(S.cpu())
    assert torch.equal(out[0], out[1])
    ref = oracle.commit_layers(layers)
    assert rel_fro(out[1].numpy().astype(np.float64), ref) <= TOL["bf16"]
