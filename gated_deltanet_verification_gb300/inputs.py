"""Seeded synthetic inputs for closed-form GDN tree verification.

This module only draws inputs: proposal trees (parent arrays in
parent-before-child order), per-node q/k/v, decay and write gates, the
pre-tree state and the accepted node per request.  It holds none of the
verification arithmetic, so both the CUDA path and the CPU oracle can be fed
from it without sharing any of the method's code.

Workloads follow the five configurations of the Bole evaluation setup
("Bole: Efficient Tree Speculation for Hybrid-Attention Language Models",
Section VI and the review's Section 5: max depth 8, top-k 4, Qwen3.5-shaped
GDN heads with d_k = d_v = 128).  The pages' datasets and drafters are not
available; random trees and Gaussian operands stand in for them.

Value recipe (all configs):
  q, k ~ N(0, 1), then L2-normalised per (node, head) over d_k;
  v ~ N(0, 1);  gamma = exp(-softplus(x)), beta = sigmoid(x), x ~ N(0, 1);
  S_pre ~ N(0, sigma^2) (sigma = 0.1 for the tiny fp32 case, else 0.05).
bf16 operands are rounded to nearest-even bf16 here and carried as float32
arrays holding exactly representable values, so every consumer sees the
identical numbers.
"""
from __future__ import annotations

import dataclasses
import heapq
from typing import List, Optional

import numpy as np

MAX_TREE_NODES = 128


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bf16 (ties to even); returns float32."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    if not np.all(np.isfinite(a)):
        raise ValueError("round_to_bf16 expects finite values")
    bits = a.view(np.uint32).copy()
    lsb = (bits >> 16) & np.uint32(1)
    bits += np.uint32(0x7FFF)
    bits += lsb  # finite inputs stay below 2**32 after the carry
    bits &= np.uint32(0xFFFF0000)
    return bits.view(np.float32)


@dataclasses.dataclass
class TreeBatch:
    """One packed forest and its per-node operands.

    Layouts (N = total nodes, token-major packed forest):
      offsets [B+1] int32, parent [N] int32 (request-local, -1 = committed root)
      q, k [N, H, dk], v [N, H, dv] float32 (bf16-exact when dtype == "bf16")
      gamma, beta [N, H] float32;  S_pre [B, H, dk, dv] float32
      accepted [B] int32 (request-local node index or -1)
    """

    name: str
    B: int
    H: int
    dk: int
    dv: int
    dtype: str  # "f32" or "bf16": the type of q/k/v and of the output O
    max_depth: int
    offsets: np.ndarray
    parent: np.ndarray
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    gamma: np.ndarray
    beta: np.ndarray
    S_pre: np.ndarray
    accepted: np.ndarray

    @property
    def N(self) -> int:
        return int(self.offsets[-1])

    @property
    def max_T(self) -> int:
        return int(np.max(np.diff(self.offsets))) if self.B > 0 else 0

    def tree_sizes(self) -> np.ndarray:
        return np.diff(self.offsets)

    def node_depths(self) -> np.ndarray:
        """Strict-ancestor count of every node (walks parent links)."""
        d = np.zeros(self.N, dtype=np.int64)
        for b in range(self.B):
            o = self.offsets[b]
            for i in range(self.offsets[b + 1] - o):
                p = self.parent[o + i]
                d[o + i] = 0 if p < 0 else d[o + p] + 1
        return d


# ---------------------------------------------------------------------------
# tree shapes
# ---------------------------------------------------------------------------

def random_parent_tree(rng: np.random.Generator, T: int, max_depth: int) -> np.ndarray:
    """Node 0 hangs off the committed root; node i > 0 picks its parent
    uniformly among earlier nodes whose depth is below max_depth."""
    if T > 1 and max_depth < 1:
        raise ValueError("a tree of more than one node needs max_depth >= 1")
    parent = np.full(T, -1, dtype=np.int32)
    depth = np.zeros(T, dtype=np.int64)
    for i in range(1, T):
        cand = np.nonzero(depth[:i] < max_depth)[0]
        p = int(cand[rng.integers(0, len(cand))])
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def chain_tree(T: int) -> np.ndarray:
    return np.arange(-1, T - 1, dtype=np.int32)


def star_tree(T: int) -> np.ndarray:
    return np.full(T, -1, dtype=np.int32)


def kary_tree(T: int, k: int = 4) -> np.ndarray:
    """Complete k-ary tree under the committed root, truncated to T nodes:
    the committed root is the heap root, so node i has parent i // k - 1."""
    return np.array([i // k - 1 for i in range(T)], dtype=np.int32)


def budgeted_forest(rng: np.random.Generator, B: int, t_lo: int, t_hi: int,
                    total_cap: int, max_depth: int, max_children: int = 4) -> List[np.ndarray]:
    """Trees chosen by greedy global selection of the highest cumulative
    draft probability (rho(child) = rho(parent) * p_edge, p ~ Dirichlet(1)
    over 1..max_children children), with per-request caps T_b ~ U[t_lo, t_hi]
    and a global cap.  Every request receives at least one node.  Ties break
    on (depth, request, creation id) so a parent always precedes its child.
    Returns request-local parent arrays in creation (topological) order."""
    caps = rng.integers(t_lo, t_hi + 1, size=B)
    # per request: list of (creation_id, parent_creation_id, depth)
    created: List[List[tuple]] = [[] for _ in range(B)]
    selected: List[List[int]] = [[] for _ in range(B)]
    heap: list = []

    def expand(b: int, parent_cid: int, parent_depth: int, parent_rho: float) -> None:
        child_depth = parent_depth + 1
        if child_depth > max_depth:
            return
        c = int(rng.integers(1, max_children + 1))
        probs = rng.dirichlet(np.ones(c))
        for p in probs:
            cid = len(created[b])
            created[b].append((cid, parent_cid, child_depth))
            heapq.heappush(heap, (-parent_rho * float(p), child_depth, b, cid))

    for b in range(B):
        expand(b, -1, -1, 1.0)
    total = 0
    # guarantee one node per request: take each request's best root child
    firsts = {}
    for item in heap:
        b = item[2]
        if b not in firsts or item < firsts[b]:
            firsts[b] = item
    for b in range(B):
        item = firsts[b]
        heap.remove(item)
        selected[b].append(item[3])
        total += 1
    heapq.heapify(heap)
    for b in range(B):
        cid = selected[b][0]
        _, _, dep = created[b][cid]
        expand(b, cid, dep, -firsts[b][0])
    while heap and total < total_cap:
        negrho, dep, b, cid = heapq.heappop(heap)
        if len(selected[b]) >= caps[b]:
            continue
        selected[b].append(cid)
        total += 1
        expand(b, cid, dep, -negrho)

    trees = []
    for b in range(B):
        sel = sorted(selected[b])
        local = {cid: i for i, cid in enumerate(sel)}
        par = np.empty(len(sel), dtype=np.int32)
        for i, cid in enumerate(sel):
            pc = created[b][cid][1]
            par[i] = -1 if pc < 0 else local[pc]
        trees.append(par)
    return trees


# ---------------------------------------------------------------------------
# operands
# ---------------------------------------------------------------------------

def _l2_normalise(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, 1e-30)


def make_batch(name: str, rng: np.random.Generator, trees: List[np.ndarray], H: int,
               dk: int, dv: int, dtype: str, max_depth: int, sigma: float,
               accept: str) -> TreeBatch:
    B = len(trees)
    sizes = np.array([len(t) for t in trees], dtype=np.int64)
    offsets = np.zeros(B + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(sizes)
    N = int(offsets[-1])
    parent = np.concatenate(trees).astype(np.int32) if N else np.zeros(0, np.int32)

    q = _l2_normalise(rng.standard_normal((N, H, dk)))
    k = _l2_normalise(rng.standard_normal((N, H, dk)))
    v = rng.standard_normal((N, H, dv))
    xg = rng.standard_normal((N, H))
    xb = rng.standard_normal((N, H))
    gamma = np.exp(-np.logaddexp(0.0, xg))
    beta = 1.0 / (1.0 + np.exp(-xb))
    S_pre = rng.standard_normal((B, H, dk, dv)) * sigma

    q = q.astype(np.float32)
    k = k.astype(np.float32)
    v = v.astype(np.float32)
    if dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    elif dtype != "f32":
        raise ValueError(dtype)

    accepted = np.full(B, -1, dtype=np.int32)
    batch = TreeBatch(name, B, H, dk, dv, dtype, max_depth, offsets, parent, q, k, v,
                      gamma.astype(np.float32), beta.astype(np.float32),
                      S_pre.astype(np.float32), accepted)
    depths = batch.node_depths()
    for b in range(B):
        o, T = offsets[b], sizes[b]
        if T == 0:
            continue
        d = depths[o:o + T]
        if accept == "deepest":
            accepted[b] = int(np.argmax(d))  # first maximum = smallest index
        elif accept == "leaf":
            par = parent[o:o + T]
            is_leaf = np.ones(T, dtype=bool)
            is_leaf[par[par >= 0]] = False
            leaves = np.nonzero(is_leaf)[0]
            accepted[b] = int(leaves[rng.integers(0, len(leaves))])
        elif accept == "uniform":
            accepted[b] = int(rng.integers(0, T))
        elif accept == "none":
            pass
        else:
            raise ValueError(accept)
    return batch


# ---------------------------------------------------------------------------
# the five configurations
# ---------------------------------------------------------------------------

CONFIG_NAMES = {
    0: "tiny fp32 single tree (B=1, H=1, dk=dv=16, T=8, depth<=3)",
    1: "single request Qwen3.5-shaped (B=1, H=16, dk=dv=128, T=32, depth<=6, bf16)",
    2: "batched packed forest (B=16, H=32, dk=dv=128, T=32, depth<=8, bf16)",
    3: "ragged budgeted batch (B=64, H=32, dk=dv=128, T_b in [8,64], N<=2048, depth<=12, bf16)",
    4: "shape extremes (B=8, H=32, dk=dv=128, T=128, bf16; chain / star / 4-ary)",
}

SHAPES_CFG4 = ("chain", "star", "4ary")


def config_batch(cfg: int, seed: Optional[int] = None, shape: str = "chain",
                 dtype: Optional[str] = None) -> TreeBatch:
    """Build one of the five workloads.  Default seed = 1000 + cfg.  dtype
    "f32" keeps q, k, v of configs 1-4 at full float32 precision (the same
    draws, not rounded to bf16)."""
    if seed is None:
        seed = 1000 + cfg
    if dtype is not None and dtype not in ("f32", "bf16"):
        raise ValueError(dtype)
    qkv = dtype or "bf16"
    rng = np.random.Generator(np.random.PCG64(seed))
    if cfg == 0:
        trees = [random_parent_tree(rng, 8, 3)]
        return make_batch("cfg0", rng, trees, 1, 16, 16, "f32", 3, 0.1, "deepest")
    if cfg == 1:
        trees = [random_parent_tree(rng, 32, 6)]
        return make_batch("cfg1", rng, trees, 16, 128, 128, qkv, 6, 0.05, "leaf")
    if cfg == 2:
        trees = [random_parent_tree(rng, 32, 8) for _ in range(16)]
        return make_batch("cfg2", rng, trees, 32, 128, 128, qkv, 8, 0.05, "uniform")
    if cfg == 3:
        trees = budgeted_forest(rng, 64, 8, 64, 2048, 12)
        return make_batch("cfg3", rng, trees, 32, 128, 128, qkv, 12, 0.05, "uniform")
    if cfg == 4:
        if shape == "chain":
            tree, md = chain_tree(128), 127
        elif shape == "star":
            tree, md = star_tree(128), 1
        elif shape == "4ary":
            tree, md = kary_tree(128, 4), 3
        else:
            raise ValueError(shape)
        trees = [tree.copy() for _ in range(8)]
        return make_batch(f"cfg4-{shape}", rng, trees, 32, 128, 128, qkv, md, 0.05,
                          "deepest")
    raise ValueError(f"unknown config {cfg}")


def random_batch(seed: int, B: int, H: int, dk: int, dv: int, sizes, max_depth: int,
                 dtype: str = "f32", sigma: float = 0.1, accept: str = "uniform",
                 shape: str = "random") -> TreeBatch:
    """Small ad-hoc batches for edge-case tests (ragged sizes, empty trees)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    trees = []
    for T in sizes:
        if T == 0:
            trees.append(np.zeros(0, dtype=np.int32))
        elif shape == "random":
            trees.append(random_parent_tree(rng, int(T), max_depth))
        elif shape == "chain":
            trees.append(chain_tree(int(T)))
        elif shape == "star":
            trees.append(star_tree(int(T)))
        elif shape == "4ary":
            trees.append(kary_tree(int(T)))
        else:
            raise ValueError(shape)
    return make_batch(f"rand{seed}", rng, trees, H, dk, dv, dtype, max_depth, sigma, accept)


def layer_batches(base: TreeBatch, n_layers: int, seed: int) -> List[TreeBatch]:
    """`n_layers` GDN layers verifying one round's packed forest: layer 0 is
    `base`; every further layer shares its offsets, parent links and accepted
    nodes and draws its own S_pre, q, k, v, gamma, beta with the same
    distributions (a layer's operands differ, the tree does not)."""
    out = [base]
    sigma = float(np.std(base.S_pre)) if base.S_pre.size else 0.05
    sizes = base.tree_sizes()
    trees = [base.parent[base.offsets[b]:base.offsets[b + 1]] for b in range(base.B)]
    for layer in range(1, n_layers):
        rng = np.random.Generator(np.random.PCG64([seed, layer]))
        lb = make_batch(f"{base.name}-layer{layer}", rng, trees, base.H, base.dk, base.dv,
                        base.dtype, base.max_depth, sigma, "none")
        lb.accepted[:] = base.accepted
        assert np.array_equal(lb.offsets, base.offsets) and len(sizes) == lb.B
        out.append(lb)
    return out


@dataclasses.dataclass
class DraftCandidates:
    """A drafter's proposal trees for B requests, packed candidate-major:
    cand_offsets [B+1], cand_parent [M] (request-local, -1 = the committed
    root, parent before child), p [M] float32 edge probabilities
    p(v | parent(v)) (each node's children sum to 1), caps [B] per-request
    node limits."""
    cand_offsets: np.ndarray
    cand_parent: np.ndarray
    p: np.ndarray
    caps: np.ndarray

    @property
    def B(self) -> int:
        return len(self.cand_offsets) - 1

    @property
    def M(self) -> int:
        return int(self.cand_offsets[-1])


def draft_candidates(seed: int, B: int, m_lo: int, m_hi: int, max_depth: int,
                     max_children: int = 4, cap_lo: int = 8, cap_hi: int = 64) -> DraftCandidates:
    """Each request's proposal tree grows level by level (breadth first, so
    parent before child): every node above max_depth gets 1..max_children
    children with Dirichlet(1) edge probabilities, until the request has
    M_b ~ U[m_lo, m_hi] candidates; caps ~ U[cap_lo, cap_hi]."""
    rng = np.random.Generator(np.random.PCG64([seed, 2]))
    offs = [0]
    parents, probs = [], []
    for _ in range(B):
        m = int(rng.integers(m_lo, m_hi + 1))
        par, pr, dep = [], [], []
        frontier = [(-1, -1)]  # (node, depth)
        while frontier and len(par) < m:
            nxt = []
            for node, d in frontier:
                if d + 1 > max_depth or len(par) >= m:
                    continue
                c = int(rng.integers(1, max_children + 1))
                ps = rng.dirichlet(np.ones(c))
                for q in ps:
                    if len(par) >= m:
                        break
                    par.append(node)
                    pr.append(q)
                    dep.append(d + 1)
                    nxt.append((len(par) - 1, d + 1))
            frontier = nxt
        parents += par
        probs += pr
        offs.append(offs[-1] + len(par))
    caps = rng.integers(cap_lo, cap_hi + 1, size=B).astype(np.int32)
    return DraftCandidates(np.asarray(offs, np.int32), np.asarray(parents, np.int32),
                           np.asarray(probs, np.float32), caps)


@dataclasses.dataclass
class Stage1Inputs:
    """Synthetic inputs of the tree-parallel convolution and gate stage for a
    packed forest: x [N, C] in-projection channels (C = H (2 dk + dv): q of
    every head, then k, then v), conv_state [B, W-1, C] (the committed
    prefix's last W-1 tokens, row W-2 the most recent), conv_w [C, W] and
    conv_b [C] (float32), gate pre-activations a, b [N, H] (float32), optional
    per-head gate scale / bias [H].  x and conv_state are bf16-representable
    float32 when dtype is "bf16"."""
    W: int
    dtype: str
    x: np.ndarray
    conv_state: np.ndarray
    conv_w: np.ndarray
    conv_b: np.ndarray
    a: np.ndarray
    b: np.ndarray
    gate_scale: Optional[np.ndarray]
    gate_bias: Optional[np.ndarray]


def stage1_inputs(batch: TreeBatch, W: int = 4, seed: int = 0, dtype: Optional[str] = None,
                  gate_terms: bool = False) -> Stage1Inputs:
    """x, conv_state ~ N(0, 1); conv_w ~ N(0, 1/W); conv_b ~ N(0, 0.1^2);
    a, b ~ N(0, 1), so that gamma = exp(-softplus(a)) and beta = sigmoid(b)
    have the pages' workload distributions.  With gate_terms, per-head
    gate scale ~ U(0.5, 2) and gate bias ~ N(0, 0.5^2)."""
    dtype = dtype or batch.dtype
    rng = np.random.Generator(np.random.PCG64([seed, 1]))
    H, dk, dv, N, B = batch.H, batch.dk, batch.dv, batch.N, batch.B
    C = H * (2 * dk + dv)
    x = rng.standard_normal((N, C)).astype(np.float32)
    st = rng.standard_normal((B, W - 1, C)).astype(np.float32)
    if dtype == "bf16":
        x, st = round_to_bf16(x), round_to_bf16(st)
    elif dtype != "f32":
        raise ValueError(dtype)
    conv_w = (rng.standard_normal((C, W)) / np.sqrt(W)).astype(np.float32)
    conv_b = (0.1 * rng.standard_normal(C)).astype(np.float32)
    a = rng.standard_normal((N, H)).astype(np.float32)
    b = rng.standard_normal((N, H)).astype(np.float32)
    gs = gb = None
    if gate_terms:
        gs = rng.uniform(0.5, 2.0, H).astype(np.float32)
        gb = (0.5 * rng.standard_normal(H)).astype(np.float32)
    return Stage1Inputs(W, dtype, x, st, conv_w, conv_b, a, b, gs, gb)


__all__ = [
    "DraftCandidates", "draft_candidates", "Stage1Inputs", "stage1_inputs", "layer_batches", "TreeBatch", "round_to_bf16", "random_parent_tree", "chain_tree", "star_tree",
    "kary_tree", "budgeted_forest", "make_batch", "config_batch", "random_batch",
    "CONFIG_NAMES", "SHAPES_CFG4", "MAX_TREE_NODES",
]
