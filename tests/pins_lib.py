"""Independent restatements used to pin the oracle (tests only).

Everything here is written from the pages' closed-form statements, not from
the oracle's node-by-node recurrence, so agreement between the two is
evidence rather than repetition:

* Lemma 1 (path-factorised state, Eq. (4)) and Lemma 2 (ancestor-masked
  system, Eq. (5)) give G, C and the cumulative decay P;
* Theorem 1 (Eq. (2)) gives O = D_P Q S_pre + C (I+G)^{-1} D_beta (V - D_P K S_pre),
  solved here with a library dense solver;
* Lemma 3 (Eq. (6)) gives (I+G)^{-1} as the finite sum of (-G)^m, m <= d;
* Eq. (10) gives the committed state from the factors (P, K, U).
All from "Bole: Efficient Tree Speculation for Hybrid-Attention Language Models".
"""
import itertools

import numpy as np


def ancestors_or_self(parent):
    """List of ancestor-or-self index sets by brute-force closure over parent links."""
    T = len(parent)
    sets = []
    for i in range(T):
        s = {i}
        changed = True
        while changed:
            changed = False
            for j in list(s):
                p = int(parent[j])
                if p >= 0 and p not in s:
                    s.add(p)
                    changed = True
        sets.append(s)
    return sets


def unit_factors(parent, q, k, gamma, beta):
    """P (cumulative decay), G and C for one (request, head) unit, float64.

    q, k: [T, dk]; gamma, beta: [T].  G_ij = beta_i (P_i/P_j) k_i.k_j for j a
    strict ancestor of i; C_ij = (P_i/P_j) q_i.k_j for j an ancestor or i."""
    T = len(parent)
    anc = ancestors_or_self(parent)
    P = np.array([np.prod([gamma[r] for r in anc[i]]) for i in range(T)])
    G = np.zeros((T, T))
    C = np.zeros((T, T))
    for i in range(T):
        for j in anc[i]:
            ratio = P[i] / P[j]
            C[i, j] = ratio * float(q[i] @ k[j])
            if j != i:
                G[i, j] = beta[i] * ratio * float(k[i] @ k[j])
    return P, G, C


def closed_form_unit(parent, S_pre, q, k, v, gamma, beta):
    """Theorem 1 for one unit via a dense library solve.  Returns O, U, P, G, C."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    S_pre = np.asarray(S_pre, np.float64)
    P, G, C = unit_factors(parent, q, k, np.asarray(gamma, np.float64),
                           np.asarray(beta, np.float64))
    T = len(parent)
    DP = np.diag(P)
    R = np.diag(np.asarray(beta, np.float64)) @ (v - DP @ k @ S_pre)
    U = np.linalg.solve(np.eye(T) + G, R)
    O = DP @ q @ S_pre + C @ U
    return O, U, P, G, C


def closed_form_batch(batch):
    """Theorem 1 over every (request, head) unit of a TreeBatch."""
    b = batch
    O = np.zeros((b.N, b.H, b.dv))
    U = np.zeros((b.N, b.H, b.dv))
    logP = np.zeros((b.N, b.H))
    for r in range(b.B):
        o0, o1 = b.offsets[r], b.offsets[r + 1]
        if o1 == o0:
            continue
        par = b.parent[o0:o1]
        for h in range(b.H):
            Oh, Uh, P, _, _ = closed_form_unit(par, b.S_pre[r, h], b.q[o0:o1, h], b.k[o0:o1, h],
                                               b.v[o0:o1, h], b.gamma[o0:o1, h],
                                               b.beta[o0:o1, h])
            O[o0:o1, h] = Oh
            U[o0:o1, h] = Uh
            logP[o0:o1, h] = np.log(P)
    return O, U, logP


def commit_from_factors(batch, U, logP, accepted=None):
    """Eq. (10): S_new = P_a S_pre + sum over the accepted path of (P_a/P_j) k_j u_j^T."""
    b = batch
    acc = b.accepted if accepted is None else accepted
    S = np.array(b.S_pre, dtype=np.float64)
    for r in range(b.B):
        a = int(acc[r])
        if a < 0:
            continue
        o0 = b.offsets[r]
        path = []
        j = a
        while j != -1:
            path.append(j)
            j = int(b.parent[o0 + j])
        for h in range(b.H):
            La = logP[o0 + a, h]
            Snew = np.exp(La) * S[r, h]
            for j in path:
                Snew = Snew + np.exp(La - logP[o0 + j, h]) * np.outer(
                    np.asarray(b.k[o0 + j, h], np.float64), U[o0 + j, h])
            S[r, h] = Snew
    return S


def all_parent_arrays(T):
    """Every valid parent-before-child array of T nodes (T! of them)."""
    choices = [range(-1, i) for i in range(T)]
    for combo in itertools.product(*choices):
        yield np.array(combo, dtype=np.int32)


def token_order_gdn(S0, q, k, v, gamma, beta):
    """Ordinary single-sequence gated delta rule (Eq. (1)), token by token."""
    S = np.array(S0, dtype=np.float64)
    outs, us = [], []
    for t in range(len(q)):
        S = gamma[t] * S
        u = beta[t] * (np.asarray(v[t], np.float64) - S.T @ np.asarray(k[t], np.float64))
        S = S + np.outer(np.asarray(k[t], np.float64), u)
        outs.append(S.T @ np.asarray(q[t], np.float64))
        us.append(u)
    return np.array(outs), np.array(us), S
