"""Invariants (b) and (c) through a real (random-init) 2-layer target (CPU only).

(b) tree-masked verification equals running each root-to-node path on its own
    through the same target (plain causal decoding);
(c) greedy acceptance commits exactly the tokens plain greedy decoding of the
    target produces.
"""
import numpy as np
import pytest

import eagle_synth as S
from oracle import tree as T
from oracle.layer import DraftWeights, fc_rows, qkv_rows, rmsnorm
from oracle.round import draft_tree
from oracle.target import TinyTarget
from oracle.verify import accept_greedy, tree_attention


@pytest.fixture(scope="module")
def setup():
    w = S.WORKLOADS["tiny_fp32"]
    seed = S.WORKLOAD_SEEDS["tiny_fp32"]
    Wt = S.draft_weights(w, seed)
    Wd = DraftWeights(Wt, w)
    tgt = TinyTarget(Wd, S.target_weights(w, seed), w)
    prefix = [int(x) for x in S.random_ints(0, w.vocab, (32,), seed, "prefix_tokens")]
    f, logits, caches = tgt.prefill(prefix)
    return w, Wd, tgt, prefix, f, logits, caches


def _tree(tokens, parents):
    anc, depth = [], []
    for s, p in enumerate(parents):
        anc.append((anc[p] if p >= 0 else 0) | (1 << s))
        depth.append(0 if p < 0 else depth[p] + 1)
    return T.Tree(list(tokens), list(parents), depth, [-1] * len(tokens), anc, {}, [1.0] * len(tokens))


def test_tree_forward_equals_each_path_decoded_alone(setup):
    w, Wd, tgt, prefix, f, logits, caches = setup
    rng = np.random.default_rng(0)
    tpl = T.template("static8")
    parents = [-1] + [0 if p < 0 else p + 1 for p in tpl.parent]
    tokens = [int(x) for x in rng.integers(0, w.vocab, len(parents))]
    tr = _tree(tokens, parents)
    f_t, lg_t, _ = tgt.forward_tree(tokens, tr.depth, tr.anc, len(prefix), caches)
    for s in range(tr.size):
        path = T.visible_table(parents)[s]
        seq = prefix + [tokens[j] for j in path]
        f_seq, lg_seq, _ = tgt.prefill(seq)
        np.testing.assert_allclose(lg_t[s], lg_seq[-1], rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(f_t[s], f_seq[-1], rtol=1e-10, atol=1e-10)


def test_single_layer_tree_attention_equals_per_path_causal_attention():
    """Same invariant for the verification attention alone, on synthetic Q/K/V: for
    every node, attention over prefix + path rows run as one causal sequence."""
    rng = np.random.default_rng(1)
    Hq, Hkv, dh, L = 8, 2, 16, 40
    tpl = T.template("static26")
    parents = [-1] + [0 if p < 0 else p + 1 for p in tpl.parent]
    tr = _tree([0] * len(parents), parents)
    Sn = tr.size
    q = rng.standard_normal((Sn, Hq, dh))
    kt, vt = rng.standard_normal((Sn, Hkv, dh)), rng.standard_normal((Sn, Hkv, dh))
    kp, vp = rng.standard_normal((L, Hkv, dh)), rng.standard_normal((L, Hkv, dh))
    out = tree_attention(q, kt, vt, kp, vp, tr.anc, 1 / np.sqrt(dh))
    G = Hq // Hkv
    for s in range(Sn):
        path = T.visible_table(parents)[s]
        K = np.concatenate([kp, kt[path]])       # the causal sequence ending at s
        V = np.concatenate([vp, vt[path]])
        for h in range(Hq):
            sc = K[:, h // G] @ q[s, h] / np.sqrt(dh)
            causal_mask = np.arange(len(K)) <= len(K) - 1     # s is the last row
            sc = np.where(causal_mask, sc, -np.inf)
            p = np.exp(sc - sc.max()); p /= p.sum()
            np.testing.assert_allclose(out[s, h], p @ V[:, h // G], rtol=1e-12, atol=1e-12)
    # a chain tree reduces to plain decode attention over prefix + chain
    chain = _tree([0] * 4, [-1, 0, 1, 2])
    oc = tree_attention(q[:4], kt[:4], vt[:4], kp, vp, chain.anc, 1 / np.sqrt(dh))
    K = np.concatenate([kp, kt[:4]]); V = np.concatenate([vp, vt[:4]])
    for s in range(4):
        sc = K[: L + s + 1, 0] @ q[s, 0] / np.sqrt(dh)
        p = np.exp(sc - sc.max()); p /= p.sum()
        np.testing.assert_allclose(oc[s, 0], p @ V[: L + s + 1, 0], rtol=1e-12)


@pytest.mark.parametrize("branch", [0, 1, 2])
def test_greedy_acceptance_reproduces_greedy_decoding(setup, branch):
    """A static8-shaped tree that hides the target's greedy continuation on one
    branch (to a depth that varies) among random tokens."""
    w, Wd, tgt, prefix, f, logits, caches = setup
    t_next = int(np.argmax(logits[-1]))
    greedy = tgt.greedy_decode(prefix + [t_next], 4)
    rng = np.random.default_rng(10 + branch)
    tpl = T.template("static8")
    parents = [-1] + [0 if p < 0 else p + 1 for p in tpl.parent]
    tokens = [t_next] + [int(x) for x in rng.integers(0, w.vocab, len(tpl.paths))]
    # plant greedy tokens along template path (branch, 0, ...) as deep as it exists
    node = {p: i + 1 for i, p in enumerate(tpl.paths)}
    path = (branch,)
    depth = 0
    while path in node:
        tokens[node[path]] = greedy[depth]
        depth += 1
        path = path + (0,)
    tr = _tree(tokens, parents)
    _, lg, _ = tgt.forward_tree(tokens, tr.depth, tr.anc, len(prefix), caches)
    a, acc_path, final = accept_greedy(tr, lg)
    committed = [tokens[s] for s in acc_path[1:]] + [final]
    assert committed == tgt.greedy_decode(prefix + [t_next], a + 1)
    assert a == depth


def test_greedy_round_with_the_drafted_tree(setup):
    """The full oracle round (draft head builds the tree from real features)."""
    w, Wd, tgt, prefix, f, logits, caches = setup
    L = len(prefix)
    t_next = int(np.argmax(logits[-1]))
    # the draft's own prefix KV: rows [f_{s-1} ; e(t_s)] at positions s = 1..L-1
    h = fc_rows(Wd, f[:L - 1], prefix[1:])
    a = rmsnorm(h, Wd.g1, w.rms_eps)
    _, dk, dv = qkv_rows(Wd, a, list(range(1, L)), w)
    inp = {"t_next": [t_next], "temps": [0.0], "philox_seed": 1, "round_id": 0,
           "prefix_len": [L], "draft_len": [L - 1], "f_last": f[L - 1][None],
           "draft_k": dk[None], "draft_v": dv[None]}
    st, tr = draft_tree(Wd, w, 0, inp)
    assert tr.size == 9 and tr.token[0] == t_next
    _, lg, _ = tgt.forward_tree(tr.token, tr.depth, tr.anc, L, caches)
    acc, path, final = accept_greedy(tr, lg)
    committed = [tr.token[s] for s in path[1:]] + [final]
    assert committed == tgt.greedy_decode(prefix + [t_next], acc + 1)
