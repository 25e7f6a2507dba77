"""Pins for the oracle's acceptance rules (CPU only).

Invariants: (a) the first draft token is accepted with probability 1 when
q == p; (c) greedy acceptance follows the target argmax chain (the pages'
worked example); (d) the accepted-token distribution equals the target
distribution, checked with exact rational arithmetic for the residual and
with chi-square tests on tiny vocabularies, with and without pruning.
"""
from fractions import Fraction

import numpy as np
import pytest
from scipy.stats import chisquare

from conftest import golden_lines
from oracle import philox
from oracle import tree as T
from oracle.sampling import draws_without_replacement, quantize
from oracle.verify import accept_greedy, accept_sampling, residual_exact


def _tree_from_parents(tokens, parents):
    anc = []
    for s, p in enumerate(parents):
        anc.append((anc[p] if p >= 0 else 0) | (1 << s))
    depth = []
    for s, p in enumerate(parents):
        depth.append(0 if p < 0 else depth[p] + 1)
    return T.Tree(list(tokens), list(parents), depth, [-1] * len(tokens), anc, {}, [1.0] * len(tokens))


def test_greedy_worked_example():
    lines = list(golden_lines("greedy_example.txt"))
    fields = dict(l.split(": ", 1) for l in lines)
    nodes = [x.split(":") for x in fields["tree"].split()]
    names = [n for n, _ in nodes]
    vocab = {n: i for i, n in enumerate(names + ["X"])}
    parents = [names.index(p) if p != "-" else -1 for _, p in nodes]
    tr = _tree_from_parents([vocab[n] for n in names], parents)
    argmax = dict(x.split(":") for x in fields["target_argmax"].split())
    logits = np.zeros((len(names), len(vocab)))
    for n, g in argmax.items():
        logits[names.index(n), vocab[g]] = 1.0
    a, path, final = accept_greedy(tr, logits)
    assert [names[s] for s in path[1:]] == fields["accepted"].split()
    assert a == 2 and final == vocab[fields["correction"]]


def test_greedy_all_accepted_gives_bonus_and_first_rejection():
    # chain R -> A -> B; target agrees everywhere -> bonus token at the leaf
    tr = _tree_from_parents([0, 1, 2], [-1, 0, 1])
    z = np.zeros((3, 5))
    z[0, 1] = z[1, 2] = z[2, 4] = 1.0
    assert accept_greedy(tr, z) == (2, [0, 1, 2], 4)
    # reject at the first layer
    z[0, 1], z[0, 3] = 0.0, 1.0
    assert accept_greedy(tr, z) == (0, [0], 3)


def _stationary_setup(rng, V, k, prune=()):
    """Root with k drawn children from q; child 0 has k drawn children of its own."""
    q_root = rng.dirichlet(np.ones(V) * 0.7)
    q_c0 = rng.dirichlet(np.ones(V) * 0.7)
    p_root = rng.dirichlet(np.ones(V) * 0.7)
    p_c0 = rng.dirichlet(np.ones(V) * 0.7)
    return q_root, q_c0, p_root, p_c0


def _run_trial(seed, V, k, q_root, q_c0, p_root, p_c0, p_leaf, prune):
    # draft: k children of the root, then k children of child 0 (all with seed `seed`)
    us = [philox.uniform_u32(seed, i, 0, philox.PURPOSE_DRAW, 0, 0) for i in range(k)]
    kids = draws_without_replacement(quantize(q_root), us)
    us = [philox.uniform_u32(seed, i, 1, philox.PURPOSE_DRAW, 0, 0) for i in range(k)]
    grand = draws_without_replacement(quantize(q_c0), us)
    child_tok = {0: kids, 1: grand}
    # retained tree: root, the root's kept children, then child 0's children
    keep = [r for r in range(k) if r not in prune]
    tokens, parents, exp_, keys = [100], [-1], [0], []
    slot_of = {}
    for r in keep:
        slot_of[(0, r)] = len(tokens)
        tokens.append(kids[r]); parents.append(0); exp_.append(1 if r == 0 else -1)
    if 0 in keep:
        for r in range(k):
            slot_of[(1, r)] = len(tokens)
            tokens.append(grand[r]); parents.append(slot_of[(0, 0)]); exp_.append(-1)
    tr = _tree_from_parents(tokens, parents)
    tr.exp = exp_
    tr.child_slot = slot_of
    p_rows = []
    for s in range(len(tokens)):
        if s == 0:
            p_rows.append(p_root)
        elif s == slot_of.get((0, 0)):
            p_rows.append(p_c0)
        else:
            p_rows.append(p_leaf)
    q_rows = {0: q_root, 1: q_c0}
    return tr, accept_sampling(tr, p_rows, q_rows, child_tok, 0, seed, 0)


def test_first_token_lemma_q_equals_p_accepts_for_every_u32():
    """Invariant (a): with q == p the test u*Q[x]*sum(P) < P[x]*sum(Q)*2^32 holds for
    every u32, because the two sides differ only by u < 2^32."""
    rng = np.random.default_rng(0)
    for _ in range(50):
        p = rng.dirichlet(np.ones(64))
        W = quantize(p)
        x = int(rng.integers(0, 64))
        while W[x] == 0:
            x = int(rng.integers(0, 64))
        S = int(W.sum())
        for u in (0, 1, (1 << 32) - 1, int(rng.integers(0, 1 << 32))):
            assert u * int(W[x]) * S < int(W[x]) * S * (1 << 32)
    # and through the full routine: a node whose only candidate was drawn from p itself
    V, hits = 6, 0
    p = rng.dirichlet(np.ones(V))
    for seed in range(300):
        us = [philox.uniform_u32(seed, 0, 0, philox.PURPOSE_DRAW, 0, 0)]
        kids = draws_without_replacement(quantize(p), us)
        tr = _tree_from_parents([100, kids[0]], [-1, 0])
        tr.exp, tr.child_slot = [0, -1], {(0, 0): 1}
        a, path, final = accept_sampling(tr, [p, p], {0: p}, {0: kids}, 0, seed, 0)
        hits += a
    assert hits == 300


def test_residual_identity_exact():
    """Page B "随机采样验证": q(x) a(x) = min(q(x), p(x)) and p - min(q, p) = max(0, p - q):
    the integer residual is exactly proportional to max(0, p - q)."""
    rng = np.random.default_rng(1)
    for _ in range(30):
        V = 7
        P = quantize(rng.dirichlet(np.ones(V)))
        Q = quantize(rng.dirichlet(np.ones(V)))
        R = residual_exact(P, Q)
        sp, sq = int(P.sum()), int(Q.sum())
        for v in range(V):
            pv, qv = Fraction(int(P[v]), sp), Fraction(int(Q[v]), sq)
            assert Fraction(R[v], sp * sq) == max(Fraction(0), pv - qv)
        # mass accounting: sum min(p, q) + sum max(0, p - q) == 1
        mins = sum(min(Fraction(int(P[v]), sp), Fraction(int(Q[v]), sq)) for v in range(V))
        assert mins + Fraction(sum(R), sp * sq) == 1


def _exact_multidraft_first_token(p, q, k):
    """Exact rational distribution of the first committed token below a node
    whose k candidates are drawn from q without replacement and tested in draw
    order against the running residual (the pages' rule, no quantisation)."""
    V = len(p)
    p = [Fraction(x) for x in p]
    q = [Fraction(x) for x in q]
    out = [Fraction(0)] * V

    def rec(P, taken, prob, i):
        if prob == 0:
            return
        Qi = [Fraction(0) if v in taken else q[v] for v in range(V)]
        sq = sum(Qi)
        if i == k or sq == 0:
            sp = sum(P)
            for v in range(V):
                out[v] += prob * P[v] / sp
            return
        sp = sum(P)
        for x in range(V):
            if Qi[x] == 0:
                continue
            px = prob * Qi[x] / sq
            a = min(Fraction(1), (P[x] / sp) / (Qi[x] / sq))
            out[x] += px * a
            res = [max(Fraction(0), P[v] / sp - Qi[v] / sq) for v in range(V)]
            if sum(res) > 0:
                rec(res, taken | {x}, px * (1 - a), i + 1)

    rec(p, frozenset(), Fraction(1), 0)
    return out


def test_multidraft_rule_is_lossless_exactly():
    """The reading that candidate i is tested against q with the earlier
    candidates removed: exact enumeration gives the target distribution."""
    rng = np.random.default_rng(2)
    for V, k in [(3, 2), (4, 3), (5, 2)]:
        p = [Fraction(int(x), 1000) for x in rng.multinomial(1000, rng.dirichlet(np.ones(V)))]
        q = [Fraction(int(x), 1000) for x in rng.multinomial(1000, rng.dirichlet(np.ones(V)))]
        p = [x / sum(p) for x in p]
        q = [x / sum(q) for x in q]
        assert _exact_multidraft_first_token(p, q, k) == p


@pytest.mark.parametrize("prune", [(), (1,), (0,)])
def test_accepted_token_distribution_chi2(prune):
    """Invariant (d): first committed token ~ p_root; second token given a
    descent into child 0 ~ p_child0; with pruned candidates too."""
    rng = np.random.default_rng(3 + len(prune))
    V, k = 5, 3
    q_root, q_c0, p_root, p_c0 = _stationary_setup(rng, V, k)
    p_leaf = rng.dirichlet(np.ones(V))
    first = np.zeros(V)
    second = np.zeros(V)
    n = 6000
    for seed in range(n):
        tr, (a, path, final) = _run_trial(seed, V, k, q_root, q_c0, p_root, p_c0, p_leaf, prune)
        toks = [tr.token[s] for s in path[1:]] + [final]
        first[toks[0]] += 1
        if a >= 1 and path[1] == tr.child_slot.get((0, 0)):
            second[toks[1]] += 1
    assert chisquare(first, p_root * n).pvalue > 1e-3
    # conditioned on descending into child 0, the next token follows p_c0
    if second.sum() > 200:
        assert chisquare(second, p_c0 * second.sum()).pvalue > 1e-3


def test_reject_all_candidates_draws_from_the_residual():
    """Force rejection of every candidate (p puts no mass on them): the final
    token never equals a rejected candidate and follows the residual."""
    V = 4
    q = np.array([0.5, 0.3, 0.1, 0.1])
    p = np.array([0.0, 0.0, 0.6, 0.4])
    counts = np.zeros(V)
    for seed in range(3000):
        kids = [0, 1]
        tr = _tree_from_parents([100, 0, 1], [-1, 0, 0])
        tr.exp, tr.child_slot = [0, -1, -1], {(0, 0): 1, (0, 1): 2}
        a, path, final = accept_sampling(tr, [p, p, p], {0: q}, {0: kids}, 0, seed, 0)
        assert a == 0
        counts[final] += 1
    assert counts[0] == counts[1] == 0
    # the pages' residual applied twice: candidate 0 against q, candidate 1 against
    # q without candidate 0 (renormalised)
    def norm(v):
        return v / v.sum()
    r1 = norm(np.maximum(0.0, p - q))
    q2 = norm(np.where(np.arange(V) == 0, 0.0, q))
    r2 = norm(np.maximum(0.0, r1 - q2))
    assert chisquare(counts[2:], r2[2:] * counts.sum()).pvalue > 1e-3
