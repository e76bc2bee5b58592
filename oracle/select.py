"""CPU oracle for device-side proposal selection and forest build -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may import this module; the CUDA library never does and shares no code with
it.  Plain Python / numpy, one candidate at a time.

What it computes ("Bole: Efficient Tree Speculation for Hybrid-Attention
Language Models", the hardware-aware budget of Section IV and its runtime
rule on the review page): every drafted candidate v of every request gets the
path score rho(v) = product over the path root..v of the drafter's edge
probabilities p(u | parent(u)); the round's proposal budget is filled with
the globally highest-scoring candidates.  Because rho(child) <= rho(parent),
each request's selection is closed under ancestors and needs no repair; the
selected nodes are then packed into the flat ragged forest (offsets, local
parent links, parent before child) that verification consumes -- the
"selection -> forest build" steps that the pages keep on the GPU.

Points the pages leave open, and the readings taken:
* rho is accumulated in float32 from the root down, rho(v) = rho(parent) * p(v)
  (rho of a root child = p), the precision the kernel uses, so both sides
  decide every comparison on identical numbers.
* Order: larger rho first; ties by smaller depth (a parent always precedes
  its child, even when p = 1), then smaller request index, then smaller
  candidate index.
* Per-request caps cap[b] (the workload's per-request tree sizes; None = no
  cap), never above 128 (a packed-forest tree holds at most 128 nodes), and,
  since a request with no proposal cannot advance, each request
  with a candidate and cap >= 1 first receives its best candidate; the rest
  of the budget goes to the best remaining candidates in the global order,
  skipping requests at their cap.  With fewer budget slots than requests,
  the reserved candidates themselves are taken in the global order.
* The packed forest lists each request's selected candidates in candidate
  order (parent before child, since candidates are), with request-local
  parent links; `src` maps each forest node to its candidate.
"""
from __future__ import annotations

import numpy as np

MAX_TREE = 128  # nodes of one packed-forest tree


def path_scores(p, cand_offsets, cand_parent):
    """(rho float32 [M], depth int32 [M]): rho(v) = rho(parent) * p(v) in
    float32, depth = number of strict candidate ancestors."""
    p = np.asarray(p, np.float32)
    M = len(p)
    rho = np.zeros(M, np.float32)
    depth = np.zeros(M, np.int32)
    for b in range(len(cand_offsets) - 1):
        o, n = int(cand_offsets[b]), int(cand_offsets[b + 1] - cand_offsets[b])
        for i in range(n):
            par = int(cand_parent[o + i])
            if par < 0:
                rho[o + i] = p[o + i]
                depth[o + i] = 0
            else:
                assert par < i, "candidates are parent-before-child"
                rho[o + i] = np.float32(rho[o + par] * p[o + i])
                depth[o + i] = depth[o + par] + 1
    return rho, depth


def select_forest(p, cand_offsets, cand_parent, budget: int, caps=None):
    """Greedy global selection and forest build.

    Returns (offsets [B+1] int32, parent [N] int32 request-local, src [N]
    int32 candidate index, rho [M] float32)."""
    cand_offsets = np.asarray(cand_offsets)
    B = len(cand_offsets) - 1
    rho, depth = path_scores(p, cand_offsets, cand_parent)
    cap = [MAX_TREE] * B if caps is None else [min(max(int(c), 0), MAX_TREE) for c in caps]
    items = []  # (-rho, depth, request, local index)
    for b in range(B):
        o, n = int(cand_offsets[b]), int(cand_offsets[b + 1] - cand_offsets[b])
        for i in range(n):
            items.append((-float(rho[o + i]), int(depth[o + i]), b, i))
    items.sort()
    chosen = [[] for _ in range(B)]
    taken = set()
    # each request's best candidate first (cap permitting), in the global order
    firsts = {}
    for it in items:
        b = it[2]
        if b not in firsts and cap[b] >= 1:
            firsts[b] = it
    total = 0
    for it in sorted(firsts.values()):
        if total >= budget:
            break
        chosen[it[2]].append(it[3])
        taken.add(it)
        total += 1
    for it in items:
        if total >= budget:
            break
        b = it[2]
        if it in taken or len(chosen[b]) >= cap[b]:
            continue
        chosen[b].append(it[3])
        taken.add(it)
        total += 1
    offsets = np.zeros(B + 1, np.int32)
    parents, src = [], []
    for b in range(B):
        o = int(cand_offsets[b])
        sel = sorted(chosen[b])
        local = {c: j for j, c in enumerate(sel)}
        for c in sel:
            pc = int(cand_parent[o + c])
            parents.append(-1 if pc < 0 else local[pc])  # KeyError = not ancestor-closed
            src.append(o + c)
        offsets[b + 1] = offsets[b] + len(sel)
    return (offsets, np.asarray(parents, np.int32), np.asarray(src, np.int32), rho)


__all__ = ["path_scores", "select_forest"]
