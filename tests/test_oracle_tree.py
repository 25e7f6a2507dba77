"""Pins for the oracle's tree construction (CPU only)."""
import itertools

import numpy as np
import pytest

from conftest import golden_lines
from oracle import tree as T


def test_visible_ancestor_table_of_the_pages():
    names, parents, want = [], [], []
    for line in golden_lines("visible_ancestors.txt"):
        left, right = line.split(":")
        node, par = left.split()
        names.append(node)
        parents.append(par)
        want.append(right.split())
    idx = {n: i for i, n in enumerate(names)}
    parent = [idx[p] if p != "-" else -1 for p in parents]
    got = T.visible_table(parent)
    assert [[names[j] for j in row] for row in got] == want
    # the oracle's bitmask form agrees with the table
    anc = []
    for s, p in enumerate(parent):
        anc.append((anc[p] if p >= 0 else 0) | (1 << s))
    for s, row in enumerate(want):
        assert {names[j] for j in range(6) if (anc[s] >> j) & 1} == set(row)


@pytest.mark.parametrize("name,rows,nodes,kmax", [
    ("chain4", [1, 1, 1, 1], 4, 1),
    ("static8", [1, 2, 1], 8, 3),
    ("static26", [1, 4, 4, 4, 1], 26, 4),
])
def test_static_templates(name, rows, nodes, kmax):
    tpl = T.template(name)
    assert tpl.layer_rows == rows and len(tpl.paths) == nodes and tpl.k_max == kmax
    # every template is a tree whose parents are listed first
    for i, p in enumerate(tpl.paths):
        assert (tpl.parent[i] < i) and (tpl.parent[i] == -1) == (len(p) == 1)


def _random_children(rng, n_exp, k, V=1000, ties=False):
    toks, qs = {}, {}
    for e in range(n_exp):
        toks[e] = list(rng.choice(V, size=k, replace=False))
        q = rng.dirichlet(np.ones(k + 3))[:k].astype(np.float32)
        if ties:
            q = np.round(q * 4) / 8 + 0.125      # few distinct values -> many ties
            q = q.astype(np.float32)
        qs[e] = [float(x) for x in q]
    return toks, qs


def _build_eagle2(rng, k, depth, m, ties=False):
    ex = T.root(5)
    toks, qs = _random_children(rng, 1, k, ties=ties)
    prev = [0]
    for layer in range(1, depth):
        prev = T.eagle2_frontier(ex, toks, qs, prev, k)
        more_t, more_q = _random_children(rng, len(ex.token), k, ties=ties)
        for e in prev:
            toks[e], qs[e] = more_t[e], more_q[e]
    return ex, toks, qs, T.eagle2_final(ex, toks, qs, m)


@pytest.mark.parametrize("ties", [False, True])
def test_eagle2_value_monotone_and_selection_connected(ties):
    rng = np.random.default_rng(7 + ties)
    for trial in range(25):
        ex, toks, qs, tr = _build_eagle2(rng, k=4, depth=4, m=12, ties=ties)
        # value(child) <= value(parent) for every expanded node (Page A §10.3 property 1)
        for e in range(1, len(ex.token)):
            assert ex.value[e] <= ex.value[ex.parent[e]]
        # the selection is a tree: each node's parent is present and shallower
        for s in range(1, tr.size):
            assert 0 <= tr.parent[s] < s and tr.depth[tr.parent[s]] == tr.depth[s] - 1
        assert tr.depth == sorted(tr.depth)
        assert tr.size == 13


def test_eagle2_rerank_is_top_m_of_the_pool_by_brute_force():
    """Enumerate every m-subset of the pool: the selection has the largest sorted
    value vector of all of them, and it is connected."""
    rng = np.random.default_rng(11)
    for trial in range(6):
        ex, toks, qs, tr = _build_eagle2(rng, k=2, depth=3, m=4)
        pool = {}
        for e in range(len(ex.token)):
            for r in range(2):
                pool[(e, r)] = ex.value[e] * qs[e][r]
        keys = list(pool)
        best = max(tuple(sorted((pool[k] for k in sub), reverse=True))
                   for sub in itertools.combinations(keys, 4))
        got = tuple(sorted((tr.value[s] for s in range(1, tr.size)), reverse=True))
        assert got == best
        exp_key = {(ex.parent[e], ex.rank[e]): e for e in range(1, len(ex.token))}
        chosen = set(tr.child_slot)
        for (e, r) in chosen:
            assert e == 0 or (ex.parent[e], ex.rank[e]) in chosen


def test_eagle2_frontier_selects_top_k_of_last_layer_only():
    rng = np.random.default_rng(12)
    ex = T.root(1)
    toks, qs = _random_children(rng, 1, 5)
    f1 = T.eagle2_frontier(ex, toks, qs, [0], 3)
    want = sorted(range(5), key=lambda r: (-qs[0][r], r))[:3]
    assert [ex.rank[e] for e in f1] == want
    assert all(ex.depth[e] == 1 and ex.parent[e] == 0 for e in f1)
    more_t, more_q = _random_children(rng, 4, 5)
    for e in f1:
        toks[e], qs[e] = more_t[e], more_q[e]
    f2 = T.eagle2_frontier(ex, toks, qs, f1, 3)
    cands = sorted(((ex.value[e] * qs[e][r], e, r) for e in f1 for r in range(5)),
                   key=lambda c: (-c[0], c[1], c[2]))[:3]
    assert [(ex.parent[e], ex.rank[e]) for e in f2] == [(e, r) for _, e, r in cands]
    # ancestor masks over expanded slots
    for e in f2:
        assert ex.anc[e] == (1 << 0) | (1 << ex.parent[e]) | (1 << e)


def test_tie_goes_to_the_shallower_node():
    # child with confidence exactly 1.0 ties its parent: the parent must win
    ex = T.root(1)
    toks = {0: [10, 11]}
    qs = {0: [0.5, 0.25]}
    f1 = T.eagle2_frontier(ex, toks, qs, [0], 2)
    toks[f1[0]] = [20, 21]
    qs[f1[0]] = [1.0, 0.0]
    toks[f1[1]] = [30, 31]
    qs[f1[1]] = [1.0, 1.0]
    tr = T.eagle2_final(ex, toks, qs, 2)
    # values: (0,0)=.5 (0,1)=.25 (e1,0)=.5 (e2,0)=.25 ...; top-2 must be the two depth-1 nodes? No:
    # (0,0)=0.5 and (e1,0)=0.5 tie -> the shallower (0,0) first, then (e1,0) at depth 2.
    assert tr.size == 3 and tr.depth == [0, 1, 2] and tr.token == [1, 10, 20]
