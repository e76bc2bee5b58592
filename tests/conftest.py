import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def make_tree_batch(parent_list, S_pre, q, k, v, gamma, beta, accepted=None, dtype="f32",
                    max_depth=127):
    """TreeBatch from explicit per-request arrays (H = 1 when 2-D operands are given)."""
    from gated_deltanet_verification_gb300.inputs import TreeBatch

    parents = [np.asarray(p, dtype=np.int32) for p in parent_list]
    B = len(parents)
    offsets = np.zeros(B + 1, dtype=np.int32)
    offsets[1:] = np.cumsum([len(p) for p in parents])
    q = np.asarray(q, dtype=np.float32)
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    gamma = np.asarray(gamma, dtype=np.float32)
    beta = np.asarray(beta, dtype=np.float32)
    S_pre = np.asarray(S_pre, dtype=np.float32)
    if q.ndim == 2:
        q, k, v = q[:, None, :], k[:, None, :], v[:, None, :]
        gamma, beta = gamma[:, None], beta[:, None]
    if S_pre.ndim == 2:
        S_pre = S_pre[None, None]
    H, dk, dv = q.shape[1], q.shape[2], v.shape[2]
    acc = np.full(B, -1, np.int32) if accepted is None else np.asarray(accepted, np.int32)
    return TreeBatch("explicit", B, H, dk, dv, dtype, max_depth, offsets,
                     np.concatenate(parents) if offsets[-1] else np.zeros(0, np.int32),
                     q, k, v, gamma, beta, S_pre, acc)


def rel_fro(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return num
    return num / den


def unit_errors(x, ref, offsets):
    """Relative Frobenius error of each (request, head) block of a node-major
    [N, H, d] tensor: {(b, h): err} for requests with nodes."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    out = {}
    for b in range(len(offsets) - 1):
        o, e = int(offsets[b]), int(offsets[b + 1])
        if e == o:
            continue
        for h in range(ref.shape[1]):
            out[(b, h)] = rel_fro(x[o:e, h], ref[o:e, h])
    return out


def state_unit_errors(x, ref):
    """Relative Frobenius error of each (request, head) state [B, H, dk, dv]."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return {(b, h): rel_fro(x[b, h], ref[b, h])
            for b in range(ref.shape[0]) for h in range(ref.shape[1])}


def row_errors(x, ref, offsets, floor=0.1):
    """Per node row (node, head) of a [N, H, d] tensor: the error norm over
    max(row norm, floor x the rms row norm of the tensor), so that rows the
    oracle makes nearly zero are held to an absolute bound at the tensor's
    scale instead of a relative one.  Returns (errors [N, H], request of each
    node [N])."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.linalg.norm(x - ref, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    rms = float(np.sqrt(np.mean(den ** 2))) if den.size else 0.0
    scale = np.maximum(den, floor * rms)
    err = np.where(scale > 0, num / np.where(scale > 0, scale, 1.0), num)
    req = np.zeros(ref.shape[0], dtype=np.int64)
    for b in range(len(offsets) - 1):
        req[int(offsets[b]):int(offsets[b + 1])] = b
    return err, req


def assert_local_parity(name, what, got, ref, offsets, tol):
    """Per-(request, head) and per-node-row bounds on a [N, H, d] output, with
    the worst (request, head, node) named on failure."""
    ue = unit_errors(got, ref, offsets)
    if ue:
        (wb, wh), worst = max(ue.items(), key=lambda kv: kv[1])
        assert worst <= tol, (f"{name}: {what} worst (request, head) = ({wb}, {wh}) "
                              f"rel err {worst:.3e} > {tol}")
    err, req = row_errors(got, ref, offsets)
    if err.size:
        n, h = np.unravel_index(int(np.argmax(err)), err.shape)
        b = int(req[n])
        local = int(n) - int(offsets[b])
        assert err[n, h] <= tol, (f"{name}: {what} worst row (request {b}, head {h}, node "
                                  f"{local}) err {err[n, h]:.3e} > {tol}")
    return max(ue.values()) if ue else 0.0, float(err.max()) if err.size else 0.0
