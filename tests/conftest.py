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
