"""CPU oracle for the tree-parallel stage 1 of a GDN layer -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may import this module; the CUDA library never does and shares no code with
it.  Plain numpy in float64, one node at a time.

What it computes ("Bole: Efficient Tree Speculation for Hybrid-Attention
Language Models", Section II-A and the fused pipeline of Section IV-C: stage
(1), tree-parallel convolution and gate preparation, fusing the convolution,
its bias, SiLU and the gates per node along parent links):

* The layer's short causal depthwise convolution of width W over the
  in-projection channels x (C = H (2 dk + dv) per token: q of every head, then
  k, then v).  In token order, y_t[c] = bias[c] + sum_w w[c][w] x_{t-W+1+w}[c].
  On a proposal tree the tokens before node i are its ancestors, nearest
  first (parent, grandparent, ...), then the committed prefix, whose last W-1
  tokens are the request's convolution state (row W-2 the most recent).
* SiLU, then q and k L2-normalised per head (the q, k of the recurrence are
  unit vectors, as in the pages' workloads); v as is.
* Gates per node and head from the pre-activations a, b:
  gamma = exp(-s_h softplus(a + c_h)), beta = sigmoid(b), with per-head scale
  s_h (default 1) and bias c_h (default 0); s = 1, c = 0 is the gate of the
  pages' workloads, gamma = exp(-softplus(x)).
* Convolution-state commit: after sampling, the request's state becomes the
  last W-1 tokens that end at the accepted node a (its path from the root,
  preceded by the old state); a = -1 leaves it unchanged.

Pins (tests/test_stage1_pins.py): a chain tree reduces to token-order
numpy.convolve; a star tree gives every node a one-token decode from the
committed state; sibling relabelling permutes the outputs; closed-form gate
values; the committed state of a chain equals the token-order window.
"""
from __future__ import annotations

import numpy as np


def _silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def window_tokens(parent_local, i: int, W: int):
    """The W tokens of node i's causal window, most recent first: node
    indices >= 0 for tree nodes, then -(s + 1) for committed-state row s
    (s = W-2 the most recent committed token)."""
    out = []
    j = i
    while len(out) < W and j >= 0:
        out.append(j)
        j = int(parent_local[j])
    s = W - 2
    while len(out) < W:
        out.append(-(s + 1))
        s -= 1
    return out


def conv_gates(x, conv_state, conv_w, conv_b, a, b, offsets, parent, H: int, dk: int, dv: int,
               gate_scale=None, gate_bias=None):
    """Stage 1 for every node of every request.

    x [N, C], conv_state [B, W-1, C], conv_w [C, W], conv_b [C] or None,
    a, b [N, H]; C = H (2 dk + dv).  Returns float64 (q [N,H,dk], k [N,H,dk],
    v [N,H,dv], gamma [N,H], beta [N,H])."""
    x = np.asarray(x, np.float64)
    st = np.asarray(conv_state, np.float64)
    w = np.asarray(conv_w, np.float64)
    N, C = x.shape
    W = w.shape[1]
    assert C == H * (2 * dk + dv) and w.shape[0] == C
    bias = np.zeros(C) if conv_b is None else np.asarray(conv_b, np.float64)
    scale = np.ones(H) if gate_scale is None else np.asarray(gate_scale, np.float64)
    gbias = np.zeros(H) if gate_bias is None else np.asarray(gate_bias, np.float64)
    y = np.zeros((N, C))
    B = len(offsets) - 1
    for r in range(B):
        o, T = int(offsets[r]), int(offsets[r + 1] - offsets[r])
        par = np.asarray(parent[o:o + T])
        for i in range(T):
            acc = bias.copy()
            for dist, tok in enumerate(window_tokens(par, i, W)):
                row = x[o + tok] if tok >= 0 else st[r, -tok - 1]
                acc += w[:, W - 1 - dist] * row
            y[o + i] = _silu(acc)
    q = y[:, :H * dk].reshape(N, H, dk)
    k = y[:, H * dk:2 * H * dk].reshape(N, H, dk)
    v = y[:, 2 * H * dk:].reshape(N, H, dv)
    q = q / np.linalg.norm(q, axis=-1, keepdims=True)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    gamma = np.exp(-scale[None, :] * _softplus(a + gbias[None, :]))
    beta = 1.0 / (1.0 + np.exp(-b))
    return q, k, v, gamma, beta


def conv_commit(conv_state, x, offsets, parent, accepted):
    """The committed convolution state [B, W-1, C] (same dtype as given):
    the last W-1 tokens ending at each request's accepted node."""
    st = np.array(conv_state, copy=True)
    B, Wm1, C = st.shape
    for r in range(B):
        a = int(accepted[r])
        if a < 0:
            continue
        o, T = int(offsets[r]), int(offsets[r + 1] - offsets[r])
        par = np.asarray(parent[o:o + T])
        toks = window_tokens(par, a, Wm1 + 1)[:Wm1]  # most recent first
        old = conv_state[r]
        for pos, tok in enumerate(toks):
            st[r, Wm1 - 1 - pos] = x[o + tok] if tok >= 0 else old[-tok - 1]
    return st


__all__ = ["conv_gates", "conv_commit", "window_tokens"]
