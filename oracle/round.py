"""One draft-and-verify round per request, composed from the oracle's steps.

Round framing (our reading of Page A §6.1 vs Page B "Advanced Token"; both
describe the same algorithm with the first draft token booked differently):
the round starts from the last verified feature f_last (position L-1) and the
already-committed token t_next at position L, which the previous round drew
from the target or residual distribution -- Page A §7.1's first draft token,
accepted with probability 1.  t_next is the tree's root; a node at depth
delta sits at position L + delta.

  draft     root row [f_last ; e(t_next)]; then each frontier row
            [f^_parent ; e(token)] (Page A §6.1 steps 2-3, Page C "从 token 自回归转向特征自回归")
  tree      static template or EAGLE-2 expand/rerank (Page A §10.3)
  verify    tree-masked attention for one target layer (Page B "Tree Attention")
  accept    greedy or recursive rejection sampling (Page B "Greedy 验证", "随机采样验证")
  commit    keep the accepted path's KV and true features; the next round
            starts from the last accepted node's true feature and the final
            token (Page A §6.2 closing remark, §12 item 3; Page B "KV Cache 必须按事务提交")

The target forward is not part of the method; its outputs are synthetic
(eagle_synth): the logits of an expanded tree node are that node's draft
logits plus N(0, 0.5^2) noise, the logits of a retained but unexpanded node
are N(0, 1), and the true features / tree Q, K, V are N(0, 1).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

from . import philox, tree as T
from .layer import (DraftWeights, attend, fc_rows, finish_rows, lm_head, qkv_rows,
                    rmsnorm, softmax, to_f64)
from .sampling import draws_without_replacement, greedy_top_k, quantize
from .verify import accept_greedy, accept_sampling, tree_attention


@dataclasses.dataclass
class RequestDraft:
    ex: T.Expanded
    f_hat: Dict[int, np.ndarray] = dataclasses.field(default_factory=dict)
    z: Dict[int, np.ndarray] = dataclasses.field(default_factory=dict)
    q: Dict[int, np.ndarray] = dataclasses.field(default_factory=dict)
    k_tree: Dict[int, np.ndarray] = dataclasses.field(default_factory=dict)
    v_tree: Dict[int, np.ndarray] = dataclasses.field(default_factory=dict)
    child_tok: Dict[int, List[int]] = dataclasses.field(default_factory=dict)
    child_q: Dict[int, List[float]] = dataclasses.field(default_factory=dict)
    layers: List[List[int]] = dataclasses.field(default_factory=list)


def select_children(z: np.ndarray, q: np.ndarray, temperature: float, k: int,
                    seed: int, request: int, e: int, round_id: int):
    """Greedy: the top-k logits (ties to the lower id).  Sampling: k draws without
    replacement from the quantised q with the round's Philox stream."""
    if temperature <= 0.0:
        toks = greedy_top_k(z, k)
    else:
        u = [philox.uniform_u32(seed, i, e, philox.PURPOSE_DRAW, request, round_id)
             for i in range(k)]
        toks = draws_without_replacement(quantize(q), u)
    return toks, [float(q[t]) if t >= 0 else 0.0 for t in toks]


def draft_step(W: DraftWeights, dims, st: RequestDraft, rows: List[int], f_last: np.ndarray,
               pos0: int, draft_k: np.ndarray, draft_v: np.ndarray, draft_len: int,
               temperature: float, k: int, seed: int, request: int, round_id: int, guide=None):
    """Run the draft head on expanded nodes ``rows`` of one request.  A
    ``guide`` (see run_round) may substitute another implementation's child
    choice for a row; the row's confidences are then this oracle's q at the
    substituted tokens."""
    ex = st.ex
    feats = np.stack([f_last if e == 0 else st.f_hat[ex.parent[e]] for e in rows])
    toks = [ex.token[e] for e in rows]
    pos = [pos0 + ex.depth[e] for e in rows]
    h = fc_rows(W, feats, toks)
    a = rmsnorm(h, W.g1, dims.rms_eps)
    q, kk, vv = qkv_rows(W, a, pos, dims)
    for i, e in enumerate(rows):
        st.k_tree[e], st.v_tree[e] = kk[i], vv[i]
    scale = 1.0 / np.sqrt(dims.head_dim)
    o = np.empty_like(q)
    for i, e in enumerate(rows):
        anc = [j for j in range(len(ex.token)) if (ex.anc[e] >> j) & 1]
        K = np.concatenate([draft_k[:draft_len], np.stack([st.k_tree[j] for j in anc])])
        V = np.concatenate([draft_v[:draft_len], np.stack([st.v_tree[j] for j in anc])])
        o[i] = attend(q[i], K, V, scale)
    f_hat = finish_rows(W, h, o, dims)
    z = lm_head(W, f_hat)
    qp = softmax(z, temperature if temperature > 0 else 1.0)
    for i, e in enumerate(rows):
        st.f_hat[e], st.z[e], st.q[e] = f_hat[i], z[i], qp[i]
        st.child_tok[e], st.child_q[e] = select_children(z[i], qp[i], temperature, k, seed,
                                                         request, e, round_id)
        if guide is not None:
            toks = guide.children(request, e, st)
            if toks is not None:
                st.child_tok[e] = [int(t) for t in toks]
                st.child_q[e] = [float(qp[i][t]) if t >= 0 else 0.0 for t in toks]
    st.layers.append(list(rows))


def _follow(choice, own):
    return own if choice is None else choice


def draft_tree(W, w, b: int, inp: dict, guide=None) -> (RequestDraft, T.Tree):
    """Draft phase + tree construction for request b (``guide``: see run_round)."""
    t_next = int(inp["t_next"][b])
    st = RequestDraft(T.root(t_next))
    temp = float(inp["temps"][b])
    seed, rid = inp["philox_seed"], inp["round_id"]
    L, Ld = inp["prefix_len"][b], inp["draft_len"][b]
    args = dict(f_last=inp["f_last"][b], pos0=L, draft_k=inp["draft_k"][b],
                draft_v=inp["draft_v"][b], draft_len=Ld, temperature=temp, seed=seed,
                request=b, round_id=rid, guide=guide)
    if w.tree == "eagle2":
        draft_step(W, w, st, [0], k=w.top_k, **args)
        prev = [0]
        for _ in range(1, w.depth):
            keys = T.eagle2_frontier_keys(st.ex, st.child_tok, st.child_q, prev, w.top_k)
            if guide is not None:
                keys = _follow(guide.frontier(b, st, prev, keys), keys)
            prev = T.expand_keys(st.ex, st.child_tok, st.child_q, keys, width=w.top_k)
            draft_step(W, w, st, prev, k=w.top_k, **args)
        keys = T.eagle2_final_keys(st.ex, st.child_tok, st.child_q, w.top_m)
        if guide is not None:
            keys = _follow(guide.final(b, st, keys), keys)
        tr = T.tree_from_keys(st.ex, st.child_tok, st.child_q, keys)
    else:
        tpl = T.template(w.tree)
        draft_step(W, w, st, [0], k=tpl.k_max, **args)
        for depth in range(1, max(tpl.depth)):
            rows = T.static_frontier(st.ex, st.child_tok, tpl, depth, st.child_q)
            draft_step(W, w, st, rows, k=tpl.k_max, **args)
        tr = T.static_final(st.ex, st.child_tok, tpl)
    return st, tr


def draft_refresh_rows(W: DraftWeights, dims, feats: np.ndarray, tokens, positions):
    """The draft layer's K/V of committed positions, from true features (Page
    B "KV Cache 必须按事务提交": after a round the drafter continues from the
    committed path; Page A §6.2 closing remark: the accepted path's true
    features replace the drafted ones).  Row i: x = [f_{p-1} ; e(t_p)] at
    position p; returns k, v [n, Hkv, dh] after RoPE, as the draft layer
    would store them for those positions."""
    h = fc_rows(W, np.asarray(feats, dtype=np.float64), list(tokens))
    a = rmsnorm(h, W.g1, dims.rms_eps)
    _, k, v = qkv_rows(W, a, list(positions), dims)
    return k, v


def synthetic_target_logits(st: RequestDraft, tr: T.Tree, noise: np.ndarray,
                            fresh: np.ndarray) -> np.ndarray:
    rows = []
    for s in range(tr.size):
        e = tr.exp[s]
        rows.append(st.z[e] + noise[s] if e >= 0 else fresh[s])
    return np.stack(rows)


def commit(tr: T.Tree, path: List[int], final: int, L: int, tree_k, tree_v, f_true):
    """Commit transaction (Page B "KV Cache 必须按事务提交"): the root and the
    accepted path become authoritative at positions L..L+a, rejected
    branches are dropped; the next round starts from the last accepted node's
    true feature and the final token."""
    a = len(path) - 1
    return {
        "kv_rows_k": np.stack([tree_k[s] for s in path]),
        "kv_rows_v": np.stack([tree_v[s] for s in path]),
        "kv_positions": list(range(L, L + a + 1)),
        "f_commit": np.stack([f_true[s] for s in path]),
        "tok_commit": [tr.token[s] for s in path] + [int(final)],
        "f_last": f_true[path[-1]].copy(),
        "t_next": int(final),
        "prefix_len": L + a + 1,
    }


def numpy_inputs(inp: dict) -> dict:
    out = {}
    for key, val in inp.items():
        out[key] = to_f64(val) if hasattr(val, "dtype") and key not in ("t_next",) else val
    out["t_next"] = [int(x) for x in to_f64(inp["t_next"])]
    return out


def run_round(W: DraftWeights, w, inp: dict, requests: Optional[List[int]] = None,
              guide=None) -> List[dict]:
    """The whole round for the listed requests (all by default).

    ``guide`` (test harness use) lets the round follow another
    implementation's discrete choices: at each decision -- a row's children,
    an EAGLE-2 frontier, the rerank, the acceptance walk -- this oracle first
    makes its own choice, then calls guide.children(b, e, st) /
    guide.frontier(b, st, prev, keys) / guide.final(b, st, keys) /
    guide.accept(b, tree, result), which return the choice to continue with
    (None or the given value keeps this oracle's own).  The arithmetic of
    every step is unchanged; only which branch is followed."""
    if "f_last" in inp and not isinstance(inp["f_last"], np.ndarray):
        inp = numpy_inputs(inp)
    res = []
    for b in (range(w.batch) if requests is None else requests):
        st, tr = draft_tree(W, w, b, inp, guide=guide)
        S = tr.size
        L = inp["prefix_len"][b]
        tl = synthetic_target_logits(st, tr, inp["tgt_noise"][b], inp["tgt_fresh"][b])
        scale = 1.0 / np.sqrt(w.head_dim)
        o = tree_attention(inp["tree_q"][b][:S], inp["tree_k"][b][:S], inp["tree_v"][b][:S],
                           inp["tgt_k"][b][:L], inp["tgt_v"][b][:L], tr.anc, scale)
        temp = float(inp["temps"][b])
        if temp <= 0.0:
            p = None
            a, path, final = accept_greedy(tr, tl)
        else:
            p = softmax(tl, temp)
            a, path, final = accept_sampling(tr, p, st.q, st.child_tok, b,
                                             inp["philox_seed"], inp["round_id"])
        if guide is not None:
            a, path, final = _follow(guide.accept(b, tr, (a, path, final)), (a, path, final))
        cm = commit(tr, path, final, L, inp["tree_k"][b], inp["tree_v"][b], inp["f_true"][b])
        cm["draft_root_k"], cm["draft_root_v"] = st.k_tree[0], st.v_tree[0]
        cm["draft_len"] = inp["draft_len"][b] + 1
        res.append(dict(draft=st, tree=tr, target_logits=tl, target_probs=p, verify_out=o,
                        accept_len=a, path=path, final=final, commit=cm))
    return res
