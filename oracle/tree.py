"""Draft trees: static templates, EAGLE-2 expansion + rerank, flattening (oracle side).

Bookkeeping used throughout (our layout; the pages fix only the rules):
  * expanded nodes -- nodes the draft head runs on -- get slots e = 0, 1, ...
    in creation order; e = 0 is the root (the already-committed token t_next);
    an EAGLE-2 expansion layer always occupies k consecutive slots (layer l
    at 1 + (l - 1) k .. l k): when fewer than k candidates exist (rows whose
    distribution ran out of mass draw fewer children), the layer's last
    slots stay inactive (token -1).  Slot numbers matter beyond bookkeeping:
    they key the uniforms of each node's draws;
  * every expanded node e has k drawn children (e, r), r = draw rank;
  * the verified tree has slot 0 = root and slots 1..m sorted by
    (depth asc, rank in the selection order asc);
  * anc[i] is a bitmask over tree slots: bit j set iff j is an ancestor of i or
    j == i (Page B "Tree Attention 如何一次验证多条路径": M_uv = 0 iff v is an
    ancestor of u or v = u).

EAGLE-2 (Page A §10.3; Page C "EAGLE-2：固定树变成上下文感知动态树"):
  value(root) = 1, value(child) = value(parent) * c_child, c = draft confidence
  q_parent(child).  Expansion: the next frontier is the top-k nodes of the
  last layer by value.  Rerank: the top-m nodes of the whole pool by value;
  ties go to the shallower node (Page A §10.3 property 2 and exercise 5),
  which keeps the selection a connected tree.  Remaining ties are broken by
  creation order (parent slot, draw rank), our reading.
"""
from __future__ import annotations

import dataclasses
import itertools
from typing import Dict, List, Optional, Sequence, Tuple

# Static templates: rank paths below the root (reading: the pages give no
# layout, only "3 forwards -> 10-token tree" and "deeper/wider on likely
# branches"; parity unpinned).
STATIC_TEMPLATES: Dict[str, List[Tuple[int, ...]]] = {
    "chain4": [(0,), (0, 0), (0, 0, 0), (0, 0, 0, 0)],
    "static8": [(0,), (1,), (2,), (0, 0), (0, 1), (1, 0), (0, 0, 0), (0, 0, 1)],
    "static26": [
        (0,), (1,), (2,), (3,),
        (0, 0), (0, 1), (0, 2), (0, 3), (1, 0), (1, 1), (2, 0), (3, 0),
        (0, 0, 0), (0, 0, 1), (0, 0, 2), (0, 1, 0), (0, 1, 1), (1, 0, 0), (2, 0, 0),
        (0, 0, 0, 0), (0, 0, 0, 1), (0, 0, 1, 0), (0, 1, 0, 0), (1, 0, 0, 0),
        (0, 0, 0, 0, 0), (0, 0, 0, 0, 1),
    ],
    # the complete ternary tree of depth 4: 3 + 9 + 27 + 81 = 120 nodes, a
    # template beyond the 63 nodes one 64-bit ancestor mask can cover
    "ternary4": [path for depth in range(1, 5) for path in itertools.product(range(3), repeat=depth)],
}


@dataclasses.dataclass
class Template:
    paths: List[Tuple[int, ...]]
    parent: List[int]        # template index of the parent, -1 = root
    rank: List[int]
    depth: List[int]
    exp_slot: List[int]      # expanded slot e of the node, -1 if it has no children
    k_max: int
    layer_rows: List[int]    # expanded nodes per depth 0..D-1

    @property
    def n_expanded(self) -> int:
        return sum(self.layer_rows)


def template(name_or_paths) -> Template:
    paths = STATIC_TEMPLATES[name_or_paths] if isinstance(name_or_paths, str) else list(name_or_paths)
    index = {p: i for i, p in enumerate(paths)}
    parent, rank, depth = [], [], []
    for p in paths:
        assert len(p) >= 1
        if len(p) > 1:
            assert p[:-1] in index and index[p[:-1]] < index[p], "parents must be listed first"
        parent.append(index[p[:-1]] if len(p) > 1 else -1)
        rank.append(p[-1])
        depth.append(len(p))
    assert depth == sorted(depth), "template must be listed by depth"
    has_child = [False] * len(paths)
    for par in parent:
        if par >= 0:
            has_child[par] = True
    exp_slot, e = [], 1
    for i in range(len(paths)):
        if has_child[i]:
            exp_slot.append(e)
            e += 1
        else:
            exp_slot.append(-1)
    D = max(depth)
    layer_rows = [1] + [sum(1 for i in range(len(paths)) if has_child[i] and depth[i] == l)
                        for l in range(1, D)]
    return Template(paths, parent, rank, depth, exp_slot, max(rank) + 1, layer_rows)


@dataclasses.dataclass
class Expanded:
    """Expanded nodes of one request (the EAGLE-2 pool's inner nodes)."""
    token: List[int] = dataclasses.field(default_factory=list)
    parent: List[int] = dataclasses.field(default_factory=list)
    rank: List[int] = dataclasses.field(default_factory=list)
    depth: List[int] = dataclasses.field(default_factory=list)
    value: List[float] = dataclasses.field(default_factory=list)
    anc: List[int] = dataclasses.field(default_factory=list)     # bitmask over e

    def add_inactive(self, depth) -> int:
        """An unused slot of an expansion layer (token -1)."""
        e = len(self.token)
        self.token.append(-1)
        self.parent.append(-1)
        self.rank.append(0)
        self.depth.append(depth)
        self.value.append(-1.0)
        self.anc.append(0)
        return e

    def add(self, token, parent, rank, depth, value) -> int:
        e = len(self.token)
        self.token.append(int(token))
        self.parent.append(parent)
        self.rank.append(rank)
        self.depth.append(depth)
        self.value.append(float(value))
        self.anc.append((self.anc[parent] if parent >= 0 else 0) | (1 << e))
        return e


def root(t_next: int) -> Expanded:
    ex = Expanded()
    ex.add(t_next, -1, 0, 0, 1.0)
    return ex


def eagle2_frontier_keys(ex: Expanded, child_tok, child_q, prev: Sequence[int], k: int) -> List[Tuple[int, int]]:
    """The expansion step's choice: among the children of the previous
    frontier, the top-k drawn children (e, r) by (value desc, parent slot asc,
    draw rank asc), in selection order."""
    cands = []
    for e in prev:
        for r, tok in enumerate(child_tok[e]):
            if tok < 0:
                continue
            cands.append((ex.value[e] * float(child_q[e][r]), e, r))
    cands.sort(key=lambda c: (-c[0], c[1], c[2]))
    return [(e, r) for _, e, r in cands[:k]]


def expand_keys(ex: Expanded, child_tok, child_q, keys: Sequence[Tuple[int, int]],
                width: Optional[int] = None) -> List[int]:
    """Append the drawn children ``keys`` = [(e, r)], in the given order, as
    expanded nodes with value(child) = value(e) * c; with ``width``, pad the
    layer with inactive slots to that many.  Returns the new active slots."""
    new = []
    depth = None
    for e, r in keys:
        v = ex.value[e] * float(child_q[e][r])
        depth = ex.depth[e] + 1
        new.append(ex.add(child_tok[e][r], e, r, depth, v))
    if width is not None:
        if depth is None:
            depth = 1 + max(d for d, t in zip(ex.depth, ex.token) if t >= 0)
        for _ in range(width - len(keys)):
            ex.add_inactive(depth)
    return new


def eagle2_frontier(ex: Expanded, child_tok, child_q, prev: Sequence[int], k: int) -> List[int]:
    """Expansion step: among the children of the previous frontier, keep the top-k
    by (value desc, parent slot asc, draw rank asc) and append them as expanded
    nodes.  Returns the new slots in selection order."""
    return expand_keys(ex, child_tok, child_q, eagle2_frontier_keys(ex, child_tok, child_q, prev, k), width=k)


def static_frontier(ex: Expanded, child_tok, tpl: Template, depth: int, child_q=None) -> List[int]:
    """Expansion step of a static template: the template's nodes at ``depth``
    that have children become expanded nodes, in template order.  A node's
    value is the product of the draft confidences along its path (Page A
    §10.3 defines it for every tree node; a static template does not select
    by it); without ``child_q`` values stay 1."""
    # map template node -> expanded slot of its parent
    new = []
    for i in range(len(tpl.paths)):
        if tpl.depth[i] != depth or tpl.exp_slot[i] < 0:
            continue
        par_e = 0 if tpl.parent[i] < 0 else tpl.exp_slot[tpl.parent[i]]
        tok = child_tok[par_e][tpl.rank[i]]
        value = 1.0 if child_q is None else ex.value[par_e] * float(child_q[par_e][tpl.rank[i]])
        e = ex.add(tok, par_e, tpl.rank[i], depth, value)
        assert e == tpl.exp_slot[i]
        new.append(e)
    return new


@dataclasses.dataclass
class Tree:
    token: List[int]
    parent: List[int]          # tree slot of the parent, -1 for the root
    depth: List[int]
    exp: List[int]             # expanded slot e of the node, -1 if never expanded
    anc: List[int]             # bitmask over tree slots
    child_slot: Dict[Tuple[int, int], int]   # (e, r) -> tree slot, for retained drawn children
    value: List[float]

    @property
    def size(self) -> int:
        return len(self.token)

    def children(self, s: int) -> List[int]:
        return [i for i in range(self.size) if self.parent[i] == s]


def _flatten(ex: Expanded, chosen: List[Tuple[int, int]], child_tok, values) -> Tree:
    """chosen: retained (e, r) keys in selection order.  Slots 1..m sorted by
    (depth asc, selection rank asc)."""
    depth_of = {key: ex.depth[key[0]] + 1 for key in chosen}
    order = sorted(range(len(chosen)), key=lambda i: (depth_of[chosen[i]], i))
    keys = [chosen[i] for i in order]
    slot_of_key = {key: 1 + j for j, key in enumerate(keys)}
    # expanded slot -> pool key it came from
    key_of_exp = {e: (ex.parent[e], ex.rank[e]) for e in range(1, len(ex.token)) if ex.token[e] >= 0}
    exp_of_key = {v: e for e, v in key_of_exp.items()}
    token, parent, depth, exp_, value = [ex.token[0]], [-1], [0], [0], [1.0]
    for key in keys:
        e, r = key
        token.append(int(child_tok[e][r]))
        if e == 0:
            parent.append(0)
        else:
            pk = key_of_exp[e]
            if pk not in slot_of_key:
                raise ValueError("selection is not connected")
            parent.append(slot_of_key[pk])
        depth.append(depth_of[key])
        exp_.append(exp_of_key.get(key, -1))
        value.append(values[key])
    anc = []
    for s in range(len(token)):
        anc.append((anc[parent[s]] if parent[s] >= 0 else 0) | (1 << s))
    return Tree(token, parent, depth, exp_, anc, dict(slot_of_key), value)


def _pool_values(ex: Expanded, child_tok, child_q) -> Dict[Tuple[int, int], float]:
    values = {}
    for e in range(len(ex.token)):
        if ex.token[e] < 0:
            continue
        for r, tok in enumerate(child_tok[e]):
            if tok >= 0:
                values[(e, r)] = ex.value[e] * float(child_q[e][r])
    return values


def eagle2_final_keys(ex: Expanded, child_tok, child_q, m: int) -> List[Tuple[int, int]]:
    """The rerank's choice: the top-m drawn children (e, r) of every expanded
    node by (value desc, depth asc, parent slot asc, draw rank asc)."""
    values = _pool_values(ex, child_tok, child_q)
    pool = sorted(values, key=lambda key: (-values[key], ex.depth[key[0]] + 1, key[0], key[1]))
    return pool[:m]


def tree_from_keys(ex: Expanded, child_tok, child_q, keys: Sequence[Tuple[int, int]]) -> Tree:
    """Flatten the retained drawn children ``keys`` (selection order)."""
    return _flatten(ex, list(keys), child_tok, _pool_values(ex, child_tok, child_q))


def eagle2_final(ex: Expanded, child_tok, child_q, m: int) -> Tree:
    """Rerank: top-m of every drawn child of every expanded node by
    (value desc, depth asc, parent slot asc, draw rank asc), then flatten."""
    return tree_from_keys(ex, child_tok, child_q, eagle2_final_keys(ex, child_tok, child_q, m))


def static_final(ex: Expanded, child_tok, tpl: Template) -> Tree:
    chosen, values = [], {}
    for i in range(len(tpl.paths)):
        par_e = 0 if tpl.parent[i] < 0 else tpl.exp_slot[tpl.parent[i]]
        key = (par_e, tpl.rank[i])
        chosen.append(key)
        values[key] = 1.0
    tree = _flatten(ex, chosen, child_tok, values)
    return tree


def visible_table(parent: Sequence[int]) -> List[List[int]]:
    """For each node, the nodes it may attend to (ancestors and itself), in
    root-to-node order."""
    out = []
    for u in range(len(parent)):
        path, v = [], u
        while v >= 0:
            path.append(v)
            v = parent[v]
        out.append(path[::-1])
    return out
