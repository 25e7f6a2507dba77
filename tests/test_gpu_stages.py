"""Stage parity on identical inputs: the GPU tree construction (root,
EAGLE-2 frontier / static expansion, rerank and flatten) and the acceptance
walk (greedy and recursive multi-candidate rejection) against the oracle,
both fed the same seeded fp32 confidences and probabilities.  With the same
inputs every discrete result is fixed, so everything is compared bit-exact:
pool tokens, parents, depths and fp64 values, the flattened tree, the
ancestor masks, and accept lengths, paths and final tokens.  No near-tie
allowance applies here.

Confidences are drawn on a coarse grid (multiples of 1/8, 1 included) so
that equal node values -- across siblings, parents and depths -- are common
and the tie-break order (value, depth, parent slot, draw rank) is exercised."""
import numpy as np
import pytest
import torch

import eagle_synth as S
from eagle_feature_level_gb300 import _binding as B
from eagle_feature_level_gb300.runtime import _p
from eagle_feature_level_gb300.workload import make_round
from oracle import tree as T
from oracle import verify as Vf
from tests.gpu_harness import mask_ints

pytestmark = pytest.mark.gpu

_SMALL = dict(d=128, n_q_heads=2, n_kv_heads=2, head_dim=64, d_ff=344, vocab=1000, batch=4, prefix_len=64,
              prefix_range=None, weight_std=0.05)
CASES = {
    "eagle2_k10_d6_m60": S.variant("7b_eagle2", name="stage_eagle2_k10", temps=(0.0, 1.0, 0.0, 0.7), **_SMALL),
    "eagle2_k4_d4_m12": S.variant("7b_eagle2", name="stage_eagle2_k4", top_k=4, depth=4, top_m=12,
                                  temps=(1.0, 0.0), **_SMALL),
    "static26": S.variant("7b_static26", name="stage_static26", temps=(0.0, 1.0), **_SMALL),
    "chain4": S.variant("7b_static26", name="stage_chain4", tree="chain4", top_k=1, depth=4, top_m=4,
                        temps=(0.0, 1.0), **_SMALL),
    # six requests, some roots cut to fewer children than k: short expansion
    # layers, whose unused slots stay inactive
    "eagle2_short_layers": S.variant("7b_eagle2", name="stage_outcomes", temps=(0.0, 0.0, 0.0, 1.0, 1.0, 0.7),
                                     **dict(_SMALL, batch=6)),
}


def _uniform(shape, seed, name):
    x = S.random_tensor(shape, seed, name).double()
    return (0.5 * (1.0 + torch.erf(x / np.sqrt(2.0)))).numpy()


def _children(w, seed, Bn, E, K, V):
    """Drawn children: k distinct tokens per expanded slot in draw order,
    fp32 confidences on the 1/8 grid, some lists cut short by -1."""
    keys = S.random_tensor((Bn, E, V), seed, "stage_child_keys").numpy()
    tok = np.argsort(keys, axis=-1, kind="stable")[..., :K].astype(np.int32)
    q = ((np.floor(_uniform((Bn, E, K), seed, "stage_child_q") * 8.0) + 1.0) / 8.0).astype(np.float32)
    cut = _uniform((Bn, E), seed, "stage_child_cut")
    k = w.top_k
    tok[..., k:] = -1
    q[..., k:] = 0.0
    for b in range(Bn):
        for e in range(E):
            if w.tree == "eagle2" and cut[b, e] < 0.1 and k > 1:   # mass ran out after the first draws
                n = 1 + int(cut[b, e] * 10 * (k - 1)) % (k - 1)
                tok[b, e, n:] = -1
                q[b, e, n:] = 0.0
    return tok, q


def _gpu_tree(eng, rd, tok, q):
    rd.c_token.copy_(torch.from_numpy(tok))
    rd.c_prob.copy_(torch.from_numpy(q))
    st, ws = eng.stream(), eng.ws.data_ptr()
    B.eagle_tree_expand_rerank(eng.ctx, rd.plan, B.PHASE_ROOT, 0, rd.B, rd.req_c, None, rd.pool_c, None, ws, st)
    for layer in range(1, rd.plan.n_layers):
        B.eagle_tree_expand_rerank(eng.ctx, rd.plan, B.PHASE_FRONTIER, layer, rd.B, rd.req_c, rd.children_c,
                                   rd.pool_c, None, ws, st)
    B.eagle_tree_expand_rerank(eng.ctx, rd.plan, B.PHASE_FINAL, 0, rd.B, rd.req_c, rd.children_c, rd.pool_c,
                               rd.tree_c, ws, st)
    torch.cuda.synchronize()
    assert B.eagle_read_device_status(eng.ctx, ws, st) == 0


def _oracle_tree(w, t_next, tok_b, q_b, n_layers):
    child_tok = [[int(x) for x in row] for row in tok_b]
    child_q = [[float(x) for x in row] for row in q_b]       # fp32 -> fp64, exact
    ex = T.root(int(t_next))
    if w.tree == "eagle2":
        prev = [0]
        for _layer in range(1, n_layers):
            prev = T.eagle2_frontier(ex, child_tok, child_q, prev, w.top_k)
        tr = T.eagle2_final(ex, child_tok, child_q, w.top_m)
    else:
        tpl = T.template(w.tree)
        for depth in range(1, n_layers):
            T.static_frontier(ex, child_tok, tpl, depth, child_q)
        tr = T.static_final(ex, child_tok, tpl)
    return ex, tr, child_tok


def _build(name):
    w = CASES[name]
    seed = 5200 if name == "eagle2_short_layers" else 5150 + sorted(CASES).index(name)
    inp = S.round_inputs(w, seed, device="cuda")
    eng, rd = make_round(w, inp)
    tok, q = _children(w, seed, rd.B, rd.E, rd.K, w.vocab)
    _gpu_tree(eng, rd, tok, q)
    t_next = inp["t_next"].cpu().numpy()
    refs = [_oracle_tree(w, t_next[b], tok[b], q[b], rd.plan.n_layers) for b in range(rd.B)]
    return w, seed, inp, eng, rd, tok, q, refs


@pytest.mark.parametrize("name", list(CASES))
def test_tree_stage_bit_exact(name):
    w, seed, inp, eng, rd, tok, q, refs = _build(name)
    L = inp["prefix_len"]
    for b, (ex, tr, _ct) in enumerate(refs):
        n = len(ex.token)
        assert rd.p_token[b, :n].tolist() == ex.token, (name, b)
        assert rd.p_parent[b, :n].tolist() == ex.parent, (name, b)
        assert rd.p_depth[b, :n].tolist() == ex.depth, (name, b)
        assert rd.p_value[b, :n].cpu().numpy().tolist() == ex.value, (name, b)     # fp64, bit-exact
        assert int(rd.t_size[b]) == tr.size, (name, b)
        s = tr.size
        assert rd.t_token[b, :s].tolist() == tr.token, (name, b)
        assert rd.t_parent[b, :s].tolist() == tr.parent, (name, b)
        assert rd.t_depth[b, :s].tolist() == tr.depth, (name, b)
        assert rd.t_exp[b, :s].tolist() == tr.exp, (name, b)
        assert mask_ints(rd.t_anc[b, :s]) == tr.anc, (name, b)
        assert rd.t_pos[b, :s].tolist() == [L[b] + dd for dd in tr.depth], (name, b)
        cs = rd.t_child_slot[b].cpu().numpy()
        for e in range(n):
            for r in range(rd.K):
                assert int(cs[e, r]) == tr.child_slot.get((e, r), -1), (name, b, e, r)


def _accept_inputs(w, seed, rd, refs, tok):
    """Target probabilities p per tree slot and draft rows q per expanded
    slot (fp32).  p near q at expanded slots, and the greedy argmax often a
    drawn child, so that walks descend."""
    Bn, Sn, E, V = rd.B, rd.S, rd.E, w.vocab
    qrows = S.random_probs(Bn * E, V, seed, "stage_q", sigma=1.5).view(Bn, E, V).numpy().astype(np.float64)
    for b in range(Bn):
        for e in range(E):
            for t in tok[b, e]:
                if t >= 0:
                    qrows[b, e, t] += 0.05
    qrows = (qrows / qrows.sum(-1, keepdims=True)).astype(np.float32)
    noise = S.random_tensor((Bn, Sn, V), seed, "stage_p_noise").numpy()
    fresh = S.random_probs(Bn * Sn, V, seed, "stage_p_fresh", sigma=1.5).view(Bn, Sn, V).numpy()
    boost = _uniform((Bn, Sn), seed, "stage_p_boost")
    p = np.zeros((Bn, Sn, V), dtype=np.float64)
    for b, (_ex, tr, _ct) in enumerate(refs):
        for s_ in range(Sn):
            e = tr.exp[s_] if s_ < tr.size else -1
            if e >= 0:
                row = qrows[b, e].astype(np.float64) * np.exp(0.3 * noise[b, s_])
                kids = [int(t) for t in tok[b, e] if t >= 0]
                if kids and boost[b, s_] < 0.7:       # the target's argmax is a drawn child
                    row[kids[int(boost[b, s_] * 10) % len(kids)]] = row.max() * 1.5
            else:
                row = fresh[b, s_].astype(np.float64)
            p[b, s_] = row / row.sum()
    p = p.astype(np.float32)
    argmax = np.argmax(p, axis=-1).astype(np.int32)        # first maximum = lowest id
    return qrows, p, argmax


@pytest.mark.parametrize("name", list(CASES))
def test_accept_stage_bit_exact(name):
    w, seed, inp, eng, rd, tok, q, refs = _build(name)
    qrows, p, argmax = _accept_inputs(w, seed, rd, refs, tok)
    temps = w.temps_for_batch()
    rd.temps.copy_(torch.tensor(temps, dtype=torch.float32))
    rd.set_sampling(inp["philox_seed"], inp["round_id"])
    rd.probs.copy_(torch.from_numpy(qrows))
    rd.target_probs.copy_(torch.from_numpy(p))
    rd.target_argmax.copy_(torch.from_numpy(argmax))
    st, ws = eng.stream(), eng.ws.data_ptr()
    B.eagle_accept_from_probs(eng.ctx, rd.plan, rd.B, rd.tree_c, rd.children_c, _p(rd.target_probs),
                              _p(rd.target_argmax), _p(rd.probs), rd.sampling_c, rd.acc_c, ws, st)
    torch.cuda.synchronize()
    assert B.eagle_read_device_status(eng.ctx, ws, st) == 0
    descended = 0
    for b, (_ex, tr, child_tok) in enumerate(refs):
        p_rows = p[b].astype(np.float64)
        if temps[b] <= 0:
            a, path, final = Vf.accept_greedy(tr, p_rows)
        else:
            a, path, final = Vf.accept_sampling(tr, p[b], qrows[b], child_tok, b, inp["philox_seed"],
                                                inp["round_id"])
        got_a = int(rd.accept_len[b])
        assert got_a == a, (name, b, got_a, a)
        assert rd.path[b, :a + 1].tolist() == list(path), (name, b)
        assert int(rd.final_token[b]) == int(final), (name, b)
        assert int(rd.last_slot[b]) == path[-1], (name, b)
        descended += a
    # the inputs make walks descend: the comparison covers more than the root
    assert descended > 0, name


OUTCOME_CASE = S.variant("7b_eagle2", name="stage_outcomes", temps=(0.0, 0.0, 0.0, 1.0, 1.0, 0.7),
                         **dict(_SMALL, batch=6))


def _peak(V, tok):
    row = np.zeros(V, dtype=np.float32)
    row[tok] = 1.0
    return row


def _path_to(tr, s):
    path = []
    while s >= 0:
        path.append(s)
        s = tr.parent[s]
    return path[::-1]


def test_accept_outcomes_on_gpu():
    """Acceptance outcomes of [B] "正确性与状态边界" each made to happen on the
    GPU by target rows that put all their mass on one token (so every test's
    result is fixed by construction), and each compared with the oracle:
    greedy rejection at the root, rejection in the middle of a path, a path
    accepted to a deepest leaf with the bonus token; under sampling a drawn
    child that rerank pruned accepted as the final token, every candidate of
    the root rejected with the final token from the residual, and a path
    accepted to a deepest leaf."""
    w = OUTCOME_CASE
    seed = 5200
    inp = S.round_inputs(w, seed, device="cuda")
    eng, rd = make_round(w, inp)
    tok, q = _children(w, seed, rd.B, rd.E, rd.K, w.vocab)
    _gpu_tree(eng, rd, tok, q)
    t_next = inp["t_next"].cpu().numpy()
    refs = [_oracle_tree(w, t_next[b], tok[b], q[b], rd.plan.n_layers) for b in range(rd.B)]
    V, Sn = w.vocab, rd.S
    qrows, p_rand, _ = _accept_inputs(w, seed, rd, refs, tok)
    p = p_rand.copy()
    expect = {}
    for b, (ex, tr, child_tok) in enumerate(refs):
        kids = {s: [c for c in range(tr.size) if tr.parent[c] == s] for s in range(tr.size)}
        drawn_tokens = lambda s: set(child_tok[tr.exp[s]]) if tr.exp[s] >= 0 else set()
        not_child = lambda s: next(t for t in range(V) if t not in drawn_tokens(s))
        deepest = max(range(tr.size), key=lambda s: (tr.depth[s], -s))
        if b in (0, 4):                         # root rejection (greedy / every sampled candidate)
            t = not_child(0)
            p[b, 0] = _peak(V, t)
            expect[b] = (0, [0], t)
        elif b == 1:                            # middle rejection after two accepted nodes
            mid = next(s for s in range(tr.size) if tr.depth[s] == 2 and kids[s])
            path = _path_to(tr, mid)
            for u, c in zip(path[:-1], path[1:]):
                p[b, u] = _peak(V, tr.token[c])
            t = not_child(mid)
            p[b, mid] = _peak(V, t)
            expect[b] = (2, path, t)
        elif b in (2, 5):                       # all accepted down to a deepest leaf, bonus token there
            path = _path_to(tr, deepest)
            for u, c in zip(path[:-1], path[1:]):
                p[b, u] = _peak(V, tr.token[c])
            p[b, deepest] = _peak(V, 11)
            expect[b] = (tr.depth[deepest], path, 11)
        else:                                   # b == 3: an accepted candidate that rerank pruned
            u, y = next((s, t) for s in range(tr.size) if tr.exp[s] >= 0
                        for r, t in enumerate(child_tok[tr.exp[s]])
                        if t >= 0 and tr.child_slot.get((tr.exp[s], r), -1) < 0)
            path = _path_to(tr, u)
            for a_, c in zip(path[:-1], path[1:]):
                p[b, a_] = _peak(V, tr.token[c])
            p[b, u] = _peak(V, y)
            expect[b] = (tr.depth[u], path, y)
    argmax = np.argmax(p, axis=-1).astype(np.int32)
    temps = w.temps_for_batch()
    rd.temps.copy_(torch.tensor(temps, dtype=torch.float32))
    rd.set_sampling(inp["philox_seed"], inp["round_id"])
    rd.probs.copy_(torch.from_numpy(qrows))
    rd.target_probs.copy_(torch.from_numpy(p))
    rd.target_argmax.copy_(torch.from_numpy(argmax))
    st, ws = eng.stream(), eng.ws.data_ptr()
    B.eagle_accept_from_probs(eng.ctx, rd.plan, rd.B, rd.tree_c, rd.children_c, _p(rd.target_probs),
                              _p(rd.target_argmax), _p(rd.probs), rd.sampling_c, rd.acc_c, ws, st)
    torch.cuda.synchronize()
    assert B.eagle_read_device_status(eng.ctx, ws, st) == 0
    for b, (_ex, tr, child_tok) in enumerate(refs):
        if temps[b] <= 0:
            want = Vf.accept_greedy(tr, p[b].astype(np.float64))
        else:
            want = Vf.accept_sampling(tr, p[b], qrows[b], child_tok, b, inp["philox_seed"], inp["round_id"])
        got_a = int(rd.accept_len[b])
        got = (got_a, rd.path[b, :got_a + 1].tolist(), int(rd.final_token[b]))
        assert got == (want[0], list(want[1]), int(want[2])), (b, got, want)
        assert got == (expect[b][0], list(expect[b][1]), expect[b][2]), (b, got, expect[b])
        assert int(rd.last_slot[b]) == got[1][-1]
    # the five outcomes all happened, under greedy and under sampling
    assert expect[0][0] == 0 and expect[4][0] == 0
    assert 0 < expect[1][0] and refs[1][1].children(expect[1][1][-1])
    assert expect[2][0] == max(refs[2][1].depth) and not refs[2][1].children(expect[2][1][-1])
    assert all(t != expect[3][2] for t in (refs[3][1].token[c] for c in refs[3][1].children(expect[3][1][-1])))
