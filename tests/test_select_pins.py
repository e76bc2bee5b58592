"""Pins for the selection oracle (path scores, global top-budget selection with
per-request caps, forest build).  Expected values come from brute force over
all feasible selections, from the closure property the pages state (a child
never outscores its parent), or from closed-form special cases.  CPU only."""
import itertools

import numpy as np
import pytest

from gated_deltanet_verification_gb300 import inputs as I
from oracle import select as S


def _tiny(seed, B=2, m=(3, 5), max_depth=3):
    return I.draft_candidates(seed, B, m[0], m[1], max_depth, max_children=3, cap_lo=1,
                              cap_hi=4)


def _keys(d):
    rho, depth = S.path_scores(d.p, d.cand_offsets, d.cand_parent)
    out = []
    for b in range(d.B):
        for i in range(d.cand_offsets[b], d.cand_offsets[b + 1]):
            out.append((-float(rho[i]), int(depth[i]), b, int(i - d.cand_offsets[b])))
    return out


def _brute_force(d, budget):
    """Reserve each request's best candidate (in key order while budget
    lasts), then the lexicographically best sorted key list among every
    subset of the rest that respects the caps -- the greedy optimum of a
    partition matroid, found here by enumeration."""
    keys = sorted(_keys(d))
    best_first = {}
    for k in keys:
        if k[2] not in best_first and d.caps[k[2]] >= 1:
            best_first[k[2]] = k
    reserved = sorted(best_first.values())[:budget]
    rest = [k for k in keys if k not in reserved]
    R = budget - len(reserved)
    counts = {b: sum(1 for k in reserved if k[2] == b) for b in range(d.B)}
    n = min(R, len(rest))
    best = None
    for size in range(n, -1, -1):
        for combo in itertools.combinations(rest, size):
            c = dict(counts)
            ok = True
            for k in combo:
                c[k[2]] += 1
                if c[k[2]] > d.caps[k[2]]:
                    ok = False
                    break
            if ok and (best is None or sorted(combo) < best):
                best = sorted(combo)
        if best is not None:
            break
    chosen = reserved + (best or [])
    return sorted((k[2], k[3]) for k in chosen)


@pytest.mark.parametrize("seed", range(12))
def test_selection_is_the_brute_force_optimum(seed):
    d = _tiny(seed)
    for budget in (1, 2, 4, 7):
        offsets, parent, src, _ = S.select_forest(d.p, d.cand_offsets, d.cand_parent, budget,
                                                  d.caps)
        got = []
        for b in range(d.B):
            for j in range(offsets[b], offsets[b + 1]):
                got.append((b, int(src[j] - d.cand_offsets[b])))
        assert sorted(got) == _brute_force(d, budget), (seed, budget)


def test_scores_follow_the_path_product():
    d = I.draft_candidates(3, 4, 20, 60, 6)
    rho, depth = S.path_scores(d.p, d.cand_offsets, d.cand_parent)
    for b in range(d.B):
        o = d.cand_offsets[b]
        for i in range(d.cand_offsets[b + 1] - o):
            prod, dep, j = 1.0, -1, i
            while j >= 0:
                prod *= float(d.p[o + j])
                dep += 1
                j = int(d.cand_parent[o + j])
            assert abs(float(rho[o + i]) - prod) <= 1e-6 * prod
            assert depth[o + i] == dep
            par = d.cand_parent[o + i]
            if par >= 0:
                assert rho[o + i] <= rho[o + par]  # monotone along every path


@pytest.mark.parametrize("seed", range(5))
def test_forest_is_closed_capped_and_fills_the_budget(seed):
    d = I.draft_candidates(seed, 16, 20, 120, 8)
    for budget in (16, 100, 400, 5000):
        offsets, parent, src, _ = S.select_forest(d.p, d.cand_offsets, d.cand_parent, budget,
                                                  d.caps)
        sizes = np.diff(offsets)
        avail = np.minimum(np.diff(d.cand_offsets), d.caps)
        assert offsets[-1] == min(budget, int(avail.sum()))
        assert np.all(sizes <= avail) and np.all(sizes >= (1 if budget >= d.B else 0))
        for b in range(d.B):
            par = parent[offsets[b]:offsets[b + 1]]
            assert all(-1 <= pp < j for j, pp in enumerate(par))  # parent before child
            cands = src[offsets[b]:offsets[b + 1]] - d.cand_offsets[b]
            assert np.all(np.diff(cands) > 0)
            for j, pp in enumerate(par):  # the local link is the candidate link
                cp = d.cand_parent[d.cand_offsets[b] + cands[j]]
                assert (pp == -1 and cp == -1) or cands[pp] == cp


def test_special_cases():
    d = I.draft_candidates(9, 5, 10, 20, 4)
    # cap 1: exactly each request's best root child
    d.caps[:] = 1
    offsets, parent, src, rho = S.select_forest(d.p, d.cand_offsets, d.cand_parent, 100, d.caps)
    assert np.all(np.diff(offsets) == 1) and np.all(parent == -1)
    for b in range(d.B):
        o, e = d.cand_offsets[b], d.cand_offsets[b + 1]
        roots = [i for i in range(o, e) if d.cand_parent[i] < 0]
        assert src[b] == max(roots, key=lambda i: (d.p[i], -i))
    # no caps, budget above the candidate count: everything
    offsets, _, src, _ = S.select_forest(d.p, d.cand_offsets, d.cand_parent, 10 ** 6, None)
    assert np.array_equal(src, np.arange(d.M))
    # all-ones probabilities: every score ties, so depth then request then index decide
    ones = np.ones_like(d.p)
    offsets, _, src, _ = S.select_forest(ones, d.cand_offsets, d.cand_parent, 3 * d.B, None)
    _, depth = S.path_scores(ones, d.cand_offsets, d.cand_parent)
    req = np.repeat(np.arange(d.B), np.diff(d.cand_offsets))
    order = sorted(range(d.M), key=lambda i: (depth[i], req[i], i))
    firsts = [min((i for i in range(d.M) if req[i] == b), key=lambda i: (depth[i], i))
              for b in range(d.B)]
    exp = set(firsts) | set([i for i in order if i not in firsts][:2 * d.B])
    assert set(src.tolist()) == exp


# ---- planted mistakes: each must fail at least one pin above ----
MUTANTS = {
    "depth_tie_reversed": ("items.append((-float(rho[o + i]), int(depth[o + i]), b, i))",
                           "items.append((-float(rho[o + i]), -int(depth[o + i]), b, i))"),
    "no_reserve": ("    for it in sorted(firsts.values()):\n        if total >= budget:",
                   "    for it in []:\n        if total >= budget:"),
    "caps_ignored": ("if it in taken or len(chosen[b]) >= cap[b]:", "if it in taken:"),
    "score_is_sum": ("rho[o + i] = np.float32(rho[o + par] * p[o + i])",
                     "rho[o + i] = np.float32(rho[o + par] + p[o + i])"),
    "score_is_edge_only": ("rho[o + i] = np.float32(rho[o + par] * p[o + i])",
                           "rho[o + i] = p[o + i]"),
    "forest_in_score_order": ("        sel = sorted(chosen[b])", "        sel = list(chosen[b])"),
}


def _pins_pass(mod) -> bool:
    saved = (S.path_scores, S.select_forest)
    try:
        S.path_scores, S.select_forest = mod.path_scores, mod.select_forest
        for t in [lambda: test_selection_is_the_brute_force_optimum(0),
                  lambda: test_selection_is_the_brute_force_optimum(5),
                  test_scores_follow_the_path_product,
                  lambda: test_forest_is_closed_capped_and_fills_the_budget(1),
                  test_special_cases]:
            try:
                t()
            except (AssertionError, KeyError):
                return False
        return True
    finally:
        S.path_scores, S.select_forest = saved


def test_unmodified_selection_oracle_passes():
    assert _pins_pass(S)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_selection_mutant_is_caught(name):
    import types
    old, new = MUTANTS[name]
    src = open(S.__file__).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType(f"select_{name}")
    exec(compile(src.replace(old, new), f"select_{name}", "exec"), mod.__dict__)
    assert not _pins_pass(mod), f"pins did not catch {name}"
